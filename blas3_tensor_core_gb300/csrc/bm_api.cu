// bm_api.cu -- host side of the C ABI declared in include/bm.h: argument checks,
// launch planning, TMA tensor-map encoding (128-byte swizzle), launches and the
// device status word.
//
// The tensor map is the host-built descriptor of "cp.async / ldmatrix ablation
// plan", section 1.2 (a rank-2 tiled map: global extents and strides, box
// extents, no interleave, hardware swizzle, zero fill out of bounds), with the
// constraints of section 1.3 (16-byte aligned global address, 128-byte box rows
// in 128-byte swizzle mode, whole-tile copies).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "bm.h"
#include "bm_gemm_kernel.cuh"
#include "bm_quant_kernel.cuh"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kGroupM = 16;

// Kernel variants: output tile (rows x BN), ring depth, CTAs per tile, k-blocks per stage.
//   kSingle256: 128 x 256 per CTA, 4 stages of one k-block (48 KB)
//   kSingle128: 128 x 128 per CTA, 3 stages of two k-blocks (64 KB; narrow outputs)
//   kPair256:   256 x 256 per CTA pair (cta_group::2), 3 stages of two k-blocks (64 KB per CTA)
// MXFP8 (the scale factors take tensor-memory columns beside the accumulators):
//   kSingle128Mx: 128 x 128 per CTA, 5 stages of one k-block (33 KB with scales)
//   kPair128Mx:   256 x 128 per CTA pair, 3 stages of two k-blocks (50 KB per CTA)
//   kPair256Mx:   256 x 256 per CTA pair, 5 stages of one k-block (33.5 KB per CTA),
//                 one accumulator (two 256-column ones would fill the tensor memory)
enum Variant {
    kSingle256 = 0, kSingle128 = 1, kPair256 = 2, kSingle128Mx = 3, kPair128Mx = 4, kPair256Mx = 5, kNumVariants = 6
};
constexpr int kVariantBN[kNumVariants] = {256, 128, 256, 128, 128, 256};
constexpr int kVariantStages[kNumVariants] = {4, 3, 3, 5, 3, 5};
constexpr int kVariantStageKBlocks[kNumVariants] = {1, 2, 2, 1, 2, 1};
constexpr int kVariantPair[kNumVariants] = {1, 1, 2, 1, 2, 2};
bool variant_scaled(int v) { return v >= kSingle128Mx; }

struct DeviceState {
    bool ready = false;
    int sm_count = 0;
    int cc_major = 0, cc_minor = 0;
    int device = -1;
    int *status = nullptr;  // one int, allocated on first use
    bool attrs_set = false;
    int max_pair_clusters = 0;     // co-resident clusters of the pair kernel
    int max_pair_clusters_mx = 0;  // same for the MXFP8 pair kernels (the smaller of the two)
};

std::mutex g_mutex;
DeviceState g_devices[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::atomic<uint32_t> g_timeout_ms{2000};
std::atomic<int> g_debug_stall{0};
std::atomic<int> g_tile_override{0};  // 0 = automatic, else 1 + Variant

template <int ELEM, int EPI = bm::EPI_FULL>
const void *variant_kernel_t(int v)
{
    if constexpr (ELEM == bm::ELEM_MXF8) {
        if (v == kSingle128Mx) return reinterpret_cast<const void *>(&bm::bm_gemm_tcgen05_kernel<128, 5, 1, ELEM, 1, EPI>);
        if (v == kPair256Mx) return reinterpret_cast<const void *>(&bm::bm_gemm_tcgen05_kernel<256, 5, 2, ELEM, 1, EPI>);
        return reinterpret_cast<const void *>(&bm::bm_gemm_tcgen05_kernel<128, 3, 2, ELEM, 2, EPI>);
    } else {
        switch (v) {
        case kSingle256: return reinterpret_cast<const void *>(&bm::bm_gemm_tcgen05_kernel<256, 4, 1, ELEM, 1, EPI>);
        case kSingle128: return reinterpret_cast<const void *>(&bm::bm_gemm_tcgen05_kernel<128, 3, 1, ELEM, 2, EPI>);
        default: return reinterpret_cast<const void *>(&bm::bm_gemm_tcgen05_kernel<256, 3, 2, ELEM, 2, EPI>);
        }
    }
}

// Kernel copies: bf16 and E4M3 operands with every epilogue path, bf16 GEMM
// copies without the SYRK diagonal path (beta == 0 and beta != 0), the E4M3
// beta == 0 one, and the MXFP8 ones (kinds 5, 6) of the MXFP8 variants.
constexpr int kNumKernelKinds = 7;

bool kind_fits(int v, int kind) { return (kind >= 5) == variant_scaled(v); }

const void *variant_kernel(int v, int kind = 0)
{
    switch (kind) {
    case 1: return variant_kernel_t<bm::ELEM_E4M3>(v);
    case 2: return variant_kernel_t<bm::ELEM_BF16, bm::EPI_STORE>(v);
    case 3: return variant_kernel_t<bm::ELEM_BF16, bm::EPI_COMBINE>(v);
    case 4: return variant_kernel_t<bm::ELEM_E4M3, bm::EPI_STORE>(v);
    case 5: return variant_kernel_t<bm::ELEM_MXF8>(v);
    case 6: return variant_kernel_t<bm::ELEM_MXF8, bm::EPI_STORE>(v);
    default: return variant_kernel_t<bm::ELEM_BF16>(v);
    }
}

// Shared memory of bf16 and E4M3 kernels is the same (k-blocks are 128 bytes of
// K); the MXFP8 variants add the scale atoms.
int variant_smem(int v)
{
    switch (v) {
    case kSingle256: return bm::KernelCfg<256, 4, 1, bm::ELEM_BF16, 1>::SMEM_BYTES;
    case kSingle128: return bm::KernelCfg<128, 3, 1, bm::ELEM_BF16, 2>::SMEM_BYTES;
    case kSingle128Mx: return bm::KernelCfg<128, 5, 1, bm::ELEM_MXF8, 1>::SMEM_BYTES;
    case kPair128Mx: return bm::KernelCfg<128, 3, 2, bm::ELEM_MXF8, 2>::SMEM_BYTES;
    case kPair256Mx: return bm::KernelCfg<256, 5, 2, bm::ELEM_MXF8, 1>::SMEM_BYTES;
    default: return bm::KernelCfg<256, 3, 2, bm::ELEM_BF16, 2>::SMEM_BYTES;
    }
}

bool fits_int32(int64_t v) { return v >= 0 && v <= 0x7FFFFFFFLL; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Once per device: the dynamic shared-memory size of every kernel copy, and how
// many clusters of the pair kernel fit at once (0: single-CTA tiles only).
// Co-resident clusters of two CTAs of a pair kernel (0 if none fit).
int pair_cluster_capacity(const DeviceState &st, int v, int kind)
{
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * (st.sm_count / 2), 1, 1);
    cfg.blockDim = dim3(bm::NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = variant_smem(v);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, variant_kernel(v, kind), &cfg) != cudaSuccess || clusters <= 0) {
        cudaGetLastError();
        clusters = 0;
    }
    return clusters;
}

bm_status init_kernel_attrs(DeviceState &st)
{
    for (int e = 0; e < kNumKernelKinds; ++e)
        for (int v = 0; v < kNumVariants; ++v)
            if (kind_fits(v, e) && cudaFuncSetAttribute(variant_kernel(v, e), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                        variant_smem(v)) != cudaSuccess)
                return BM_ERR_CUDA;
    st.max_pair_clusters = pair_cluster_capacity(st, kPair256, 0);
    st.max_pair_clusters_mx =
        std::min(pair_cluster_capacity(st, kPair128Mx, 5), pair_cluster_capacity(st, kPair256Mx, 5));
    st.attrs_set = true;
    return BM_OK;
}

// Current device, checked for compute capability 10.3, with the one-time set-up
// of its state (tensor-map encoder, kernel attributes). With `alloc_status` the
// device status word is allocated on first use; without it (the allocation-free
// entry point) nothing is allocated and the word is used only if it exists.
bm_status device_state(DeviceState **out, bool alloc_status = true)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return BM_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState &st = g_devices[dev];
    if (!st.ready) {
        cudaDeviceProp prop;
        if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return BM_ERR_CUDA;
        st.sm_count = prop.multiProcessorCount;
        st.cc_major = prop.major;
        st.cc_minor = prop.minor;
        st.device = dev;
        st.ready = true;
    }
    if (st.cc_major != 10 || st.cc_minor != 3) return BM_ERR_ARCH;
    if (g_encode == nullptr) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || fn == nullptr)
            return BM_ERR_CUDA;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    if (alloc_status && st.status == nullptr) {
        if (cudaMalloc(&st.status, sizeof(int)) != cudaSuccess) return BM_ERR_CUDA;
        if (cudaMemset(st.status, 0, sizeof(int)) != cudaSuccess) return BM_ERR_CUDA;
    }
    if (!st.attrs_set) {
        const bm_status a = init_kernel_attrs(st);
        if (a != BM_OK) return a;
    }
    *out = &st;
    return BM_OK;
}

int sm_count_or_default()
{
    int dev = -1;
    if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < kMaxDevices) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0) return n;
    }
    cudaGetLastError();
    return 152;  // GB300
}

// rank-2 tensor map of 2-byte (bf16) or 1-byte (E4M3, copied as bytes)
// elements: inner (contiguous) extent, outer extent, row pitch in elements.
bool encode_operand_2d(CUtensorMap *map, const void *base, int elem, int64_t inner, int64_t outer, int64_t ld,
                       uint32_t box_inner, uint32_t box_outer)
{
    const cuuint64_t esz = elem == bm::ELEM_E4M3 ? 1u : 2u;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(std::max<int64_t>(inner, 1)),
                          static_cast<cuuint64_t>(std::max<int64_t>(outer, 1))};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * esz};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, elem == bm::ELEM_E4M3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                          const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool encode_bf16_2d(CUtensorMap *map, const void *base, int64_t inner, int64_t outer, int64_t ld,
                    uint32_t box_inner, uint32_t box_outer)
{
    return encode_operand_2d(map, base, bm::ELEM_BF16, inner, outer, ld, box_inner, box_outer);
}

// Map of C for the epilogue's TMA copies: box of 128 bytes (64 bf16 or 32 fp32
// columns) x `rows` rows, 128-byte swizzle (the staging layout the epilogue
// writes). 32 rows: one warp's stores (beta == 0); 128 rows: one CTA's rows,
// loaded and stored by a half of the epilogue (beta != 0).
// No map when a row of C (n elements) does not end on a 16-byte boundary: a
// tiled TMA store clips the innermost dimension only to whole 16-byte units, so
// the last box of a row would also write the columns from n up to the next
// boundary (measured: fp32 C with n = 2162 had columns 2162 and 2163 of its
// TMA-stored tiles overwritten). Such calls store C with masked plain stores.
bool encode_c_tile(CUtensorMap *map, void *C, bm_ctype ct, int64_t m, int64_t n, int64_t ldc, uint32_t rows)
{
    const cuuint64_t esz = ct == BM_C_BF16 ? 2u : 4u;
    if ((static_cast<cuuint64_t>(n) * esz) % 16u != 0) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(n), static_cast<cuuint64_t>(m)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ldc) * esz};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / esz), rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, ct == BM_C_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                          2, C, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Map of the fp32 partial slots [slots * tile rows][tile columns] for the
// epilogue's per-warp TMA stores: box 32 x 32, 128-byte swizzle.
bool encode_slots(CUtensorMap *map, void *partial, int64_t rows, int64_t cols)
{
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 4u};
    cuuint32_t box[2] = {32u, 32u};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, partial, dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Map of an MXFP8 scale array: ceil(rows / 128) x ceil(k / 128) atoms of 512
// bytes, atom (row block, k-block) at ((row block) * ceil(k / 128) + k-block) * 512,
// seen as a 4-D tensor of bytes (256, 2, k-block, row block) so that one box brings
// `kps` k-blocks of `row_blocks` row blocks (atoms land in the order row block,
// k-block). Boxes past the last k-block or row block read zeros.
bool encode_scales(CUtensorMap *map, const void *sf, int64_t rows, int64_t k, int kps, int row_blocks)
{
    const int64_t katoms = ceil_div(k, 128);
    cuuint64_t dims[4] = {256, 2, static_cast<cuuint64_t>(katoms), static_cast<cuuint64_t>(ceil_div(rows, 128))};
    cuuint64_t strides[3] = {256, static_cast<cuuint64_t>(bm::SF_ATOM_BYTES),
                             static_cast<cuuint64_t>(katoms * bm::SF_ATOM_BYTES)};
    cuuint32_t box[4] = {256, 2, static_cast<cuuint32_t>(kps), static_cast<cuuint32_t>(row_blocks)};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void *>(sf), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Operand tile maps. K-major: box 64 (k) x rows; M/N-major: box 64 (m or n) x 64 (k).
bool encode_operand(CUtensorMap *map, const void *base, bool mn_major, int64_t rows, int64_t k, int64_t ld,
                    uint32_t tile_rows)
{
    if (mn_major) return encode_bf16_2d(map, base, rows, k, ld, 64, 64);
    return encode_bf16_2d(map, base, k, rows, ld, 64, tile_rows);
}

// Stage box of one operand (replaces *map on success): a 3-D map whose single
// copy brings this CTA's `rows` rows for all `kps` k-blocks of a stage, in the
// kernel's stage layout. K-major operand [mn][k]: dims (k within a k-block,
// row, k-block), strides (ld, one k-block); needs K to be whole k-blocks so no
// row's copy runs past its K. M/N-major operand [k][mn]: dims (m or n within a
// 64-wide chunk, k, chunk), strides (ld, 128 bytes); needs whole chunks. The
// middle dimension has the largest stride, which the encoder accepts. Returns
// false (map untouched) when the shape does not qualify or nothing is gained
// over the 2-D boxes (one k-block, one chunk).
bool encode_stage_box(CUtensorMap *map, const void *base, int elem, bool mn_major, int64_t mn, int64_t k, int64_t ld,
                      int rows, int kps)
{
    const int64_t esz = elem == bm::ELEM_E4M3 ? 1 : 2;
    const int64_t kb_elems = bm::kblock_elems(elem);
    CUtensorMap m;
    cuuint64_t dims[3], strides[2];
    cuuint32_t box[3];
    if (mn_major) {
        if (elem != bm::ELEM_BF16 || mn % 64 != 0 || (kps == 1 && rows == 64)) return false;
        dims[0] = 64;
        dims[1] = static_cast<cuuint64_t>(k);
        dims[2] = static_cast<cuuint64_t>(mn / 64);
        strides[0] = static_cast<cuuint64_t>(ld * esz);
        strides[1] = 128;
        box[0] = 64;
        box[1] = static_cast<cuuint32_t>(64 * kps);
        box[2] = static_cast<cuuint32_t>(rows / 64);
    } else {
        if (kps == 1 || k % kb_elems != 0) return false;
        dims[0] = static_cast<cuuint64_t>(kb_elems);
        dims[1] = static_cast<cuuint64_t>(mn);
        dims[2] = static_cast<cuuint64_t>(k / kb_elems);
        strides[0] = static_cast<cuuint64_t>(ld * esz);
        strides[1] = static_cast<cuuint64_t>(kb_elems * esz);
        box[0] = static_cast<cuuint32_t>(kb_elems);
        box[1] = static_cast<cuuint32_t>(rows);
        box[2] = static_cast<cuuint32_t>(kps);
    }
    cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = g_encode(&m, elem == bm::ELEM_E4M3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                                3, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    *map = m;
    return true;
}

struct Plan {
    int variant = kSingle256;
    int tile_m = bm::CTA_M, bn = 256, stages = 4, pair = 1;
    int64_t tiles_m = 0, tiles_n = 0, num_tiles = 0;
    int64_t full_tiles = 0, num_units = 0;  // whole tiles first; the rest are split k_splits ways
    int k_splits = 1, kb_per_split = 0, kb_total = 0;
    int n_split = 1;         // 2: the tiles after full_tiles run as two N halves each
    int ctas = 0;
    int fixup = 0;           // split tiles reduced inside the kernel (no reduce kernel)
    size_t slot_bytes = 0;   // partial slots at the start of the workspace; fixup counters follow
    size_t ws_bytes = 0;
};

// Largest workspace a tail split may ask for (the full-GPU split of small
// outputs is not capped).
constexpr size_t kTailSplitMaxBytes = 16u << 20;


void set_variant(Plan &pl, int v)
{
    pl.variant = v;
    pl.bn = kVariantBN[v];
    pl.stages = kVariantStages[v];
    pl.pair = kVariantPair[v];
    pl.tile_m = bm::CTA_M * pl.pair;
}

// Tiles of the SYRK schedule: one across the diagonal per tile row, then the
// tiles inside the triangle (closed forms shared with the kernel).
int64_t syrk_tile_count(int mode, int64_t tiles_m, int64_t tiles_n, int tile_m, int bn)
{
    if (tile_m == 256) return tiles_m + bm::syrk_inside_before<256, 256>(mode, tiles_m, tiles_n);
    if (bn == 128) return tiles_m + bm::syrk_inside_before<128, 128>(mode, tiles_m, tiles_n);
    return tiles_m + bm::syrk_inside_before<128, 256>(mode, tiles_m, tiles_n);
}

void syrk_coords(int mode, int64_t tiles_m, int64_t tiles_n, int tile_m, int bn, int64_t t, int64_t &tm, int64_t &tn)
{
    if (tile_m == 256) bm::syrk_tile_coords<256, 256>(mode, tiles_m, tiles_n, t, tm, tn);
    else if (bn == 128) bm::syrk_tile_coords<128, 128>(mode, tiles_m, tiles_n, t, tm, tn);
    else bm::syrk_tile_coords<128, 256>(mode, tiles_m, tiles_n, t, tm, tn);
}

// Persistent grid: one CTA (or CTA pair) per SM (pair of SMs), never more than the work units.
void size_grid(Plan &pl, int sms, int pair_clusters)
{
    pl.num_units = pl.full_tiles + (pl.num_tiles - pl.full_tiles) * (pl.n_split > 1 ? pl.n_split : pl.k_splits);
    if (pl.pair == 2) pl.ctas = static_cast<int>(2 * std::min<int64_t>(pl.num_units, pair_clusters));
    else pl.ctas = static_cast<int>(std::min<int64_t>(pl.num_units, sms));
}

// Split the last `split_tiles` tiles of the unit order `want` ways (or fewer)
// along K, if each part keeps >= 4 k-blocks, the partial slots fit `budget`,
// and the mainloop time it saves is at least `min_gain_us`. One 64-deep
// k-block of a tile takes 4 MMAs of 128 tensor-core cycles, about 0.26 us at
// 2 GHz. Summing the partials costs a few us: a second kernel when every tile
// is split (kSplitMinGainUs), extra epilogue work inside the kernel for a tail
// split. Measured for tail splits: with beta == 0 a 3.5 us gain pays (4096^2 x
// 2048 and the 5120^2 x 2048 TN GEMM ran 9 % and 5 % faster split), 2 us does
// not (4096^2 x 1024 ran slower); with beta != 0 the split units' combine with
// C makes 3.5 us lose (dW 5120^2 x 2048 75.3 -> 81.5 us), so it keeps 6 us.
constexpr double kKBlockUs = 0.256;
constexpr double kSplitMinGainUs = 6.0;
constexpr double kTailSplitMinGainUsBeta0 = 3.5;
// At most this many K splits when every tile is split. Measured on the 8 tiles
// (128 x 256) of a 512^2 output: 512^2 x 4096 ran 14.9 us with 16 splits, 12.2
// with 13 (what this cap gives) and 12.5 with 11; 512^2 x 8192 17.2 us with 19
// splits, 16.7 with 16, 14.2 with 13 and 14.4 with 12. More splits shorten each
// unit's mainloop but write and re-read more fp32 partial tiles.
constexpr int64_t kMaxAllSplits = 14;
// BF16 GEMMs of at most this many 64-deep k-blocks (K <= 320) run on single-SM
// 128 x 256 tiles rather than 256 x 256 SM-pair tiles. Measured, pair -> single:
// 4096^2 x 128 / 256 / 320 13.9 / 15.3 / 16.4 -> 10.9 / 13.3 / 15.3 us; 8192^2 x 256
// 45.3 -> 37.2 us; 2048^2 x 256 8.1 -> 6.6 us; 8192 x 4096 x 256 23.3 -> 20.6 us.
// From K = 384 on the pair tiles are faster (4096^2 x 384 16.8 vs 17.1 us, x 512
// 18.1 vs 19.8 us, 8192^2 x 512 50.2 vs 58.6 us).
constexpr int64_t kShortKBlocks = 5;

void try_split(Plan &pl, int64_t split_tiles, int64_t want, size_t budget, double min_gain_us)
{
    const size_t slot_bytes = static_cast<size_t>(pl.tile_m) * pl.bn * sizeof(float);
    want = std::min<int64_t>(want, pl.kb_total / 4);
    while (want > 1) {
        const int per = static_cast<int>(ceil_div(pl.kb_total, want));
        const int splits = static_cast<int>(ceil_div(pl.kb_total, per));
        // With whole tiles to run after them, split units go first and reduce in
        // the kernel (the sums hide behind the next mainloops; one 8-byte counter
        // per epilogue warp region follows the slots); when every tile is split,
        // the reduce kernel spreads the sums over the GPU.
        const bool fixup = split_tiles < pl.num_tiles;
        const size_t slots = static_cast<size_t>(splits) * static_cast<size_t>(split_tiles) * slot_bytes;
        const size_t need =
            slots + (fixup ? static_cast<size_t>(split_tiles) * pl.pair * bm::NUM_EPI_WARPS * 8u : 0u);
        const double gain_us = kKBlockUs * (pl.kb_total - per);
        if (splits > 1 && need <= budget && gain_us >= min_gain_us) {
            pl.k_splits = splits;
            pl.kb_per_split = per;
            pl.full_tiles = pl.num_tiles - split_tiles;
            pl.slot_bytes = slots;
            pl.ws_bytes = need;
            pl.fixup = fixup ? 1 : 0;
            return;
        }
        --want;
    }
}

// Pair tiles (256 x 256 on two SMs) whenever they alone can occupy at least half
// of the SM pairs; otherwise 128-row tiles on single SMs (more, smaller tiles).
// beta_nonzero: the call combines with C (tail splits then need a larger gain,
// as do plain E4M3 ones: a split of the 4096^3 E4M3 tail measured slower; the
// MXFP8 4096^3 tail split two ways took it from 66.1 to 62.8 us).
Plan plan_gemm(int64_t m, int64_t n, int64_t k, size_t ws_bytes, int sms, int pair_clusters,
               int elem = bm::ELEM_BF16, bool beta_nonzero = false)
{
    Plan pl;
    const int forced = g_tile_override.load() - 1;
    if (elem == bm::ELEM_MXF8) {
        // MXFP8: 256 x 256 tiles on SM pairs when those tiles alone fill half the
        // pairs, else 256 x 128 pair tiles if those do, else 128 x 128 tiles on
        // single SMs (overrides: 1 the single-SM tiles, 2 the 256 x 128 pair, 3 the
        // 256 x 256 pair)
        const int64_t wide_tiles = ceil_div(m, 256) * ceil_div(n, 256);
        const int64_t narrow_tiles = ceil_div(m, 256) * ceil_div(n, 128);
        static const int kMxForced[3] = {kSingle128Mx, kPair128Mx, kPair256Mx};
        if (forced >= 0) set_variant(pl, pair_clusters > 0 ? kMxForced[forced] : kSingle128Mx);
        else if (pair_clusters > 0 && m > bm::CTA_M && n > 128 && wide_tiles * 2 >= pair_clusters)
            set_variant(pl, kPair256Mx);
        else if (pair_clusters > 0 && m > bm::CTA_M && narrow_tiles * 2 >= pair_clusters) set_variant(pl, kPair128Mx);
        else set_variant(pl, kSingle128Mx);
    } else {
        const int64_t pair_tiles = ceil_div(m, 256) * ceil_div(n, 256);
        // BF16 with at most kShortKBlocks k-blocks per tile takes single-SM tiles:
        // with so few k-blocks the pair's cross-SM handshakes cost more than its
        // smaller operand traffic saves.
        const bool short_k = elem == bm::ELEM_BF16 && ceil_div(std::max<int64_t>(k, 1), bm::TILE_K) <= kShortKBlocks;
        if (forced >= 0 && (forced != kPair256 || pair_clusters > 0)) set_variant(pl, forced);
        else if (pair_clusters > 0 && !short_k && m > bm::CTA_M && n > 128 && pair_tiles * 2 >= pair_clusters)
            set_variant(pl, kPair256);
        else set_variant(pl, n <= 128 ? kSingle128 : kSingle256);
    }
    pl.tiles_m = ceil_div(m, pl.tile_m);
    pl.tiles_n = ceil_div(n, pl.bn);
    pl.num_tiles = pl.tiles_m * pl.tiles_n;
    pl.full_tiles = pl.num_tiles;
    pl.kb_total = static_cast<int>(ceil_div(std::max<int64_t>(k, 1), bm::kblock_elems(elem)));
    pl.kb_per_split = pl.kb_total;
    const int64_t slots = pl.pair == 2 ? pair_clusters : sms;
    if (slots > 0 && pl.kb_total >= 8) {
        if (pl.num_tiles * 2 <= slots) {
            // Too few tiles to fill half the GPU: split every tile along K.
            try_split(pl, pl.num_tiles, std::min(kMaxAllSplits, ceil_div(slots, pl.num_tiles)), ws_bytes,
                      kSplitMinGainUs);
        } else {
            // The last wave is at most half full: split its tiles along K over the idle slots.
            const int64_t tail = pl.num_tiles % slots;
            if (tail > 0 && tail * 2 <= slots) {
                try_split(pl, tail, slots / tail, std::min(ws_bytes, kTailSplitMaxBytes),
                          elem != bm::ELEM_E4M3 && !beta_nonzero ? kTailSplitMinGainUsBeta0 : kSplitMinGainUs);
                // No K split: run each tail tile as two N halves on two SM pairs
                // (256 x 256 bf16 or E4M3 pair tiles), with no partial sums. E4M3
                // 4096^3: 46.8 -> 45.5 us.
                if (pl.k_splits == 1 && pl.variant == kPair256 &&
                    (elem == bm::ELEM_BF16 || elem == bm::ELEM_E4M3)) {
                    pl.n_split = 2;
                    pl.full_tiles = pl.num_tiles - tail;
                }
            }
        }
    }
    size_grid(pl, sms, pair_clusters);
    return pl;
}

// SYRK / SYR2K: tiles touching the triangle. SYR2K runs both products through
// one accumulator, and its A and B maps serve in both operand roles, so it
// needs the variants whose A and B tiles have the same 128 rows.
// The split rules are those of GEMM: every tile is split along K (at most
// kMaxAllSplits ways) when the triangle's tiles cannot fill half the GPU (a
// second kernel sums the partials),
// and the tiles of an at most half-full last wave when that saves at least 6 us
// (summed inside the kernel; SYRK tiles always take the full epilogue).
Plan plan_syrk(int mode, int64_t n, int64_t k, size_t ws_bytes, int sms, int pair_clusters, bool two_products = false)
{
    Plan pl;
    const int64_t tiles = ceil_div(n, 256);
    const int single = two_products ? kSingle128 : kSingle256;
    int forced = g_tile_override.load() - 1;
    if (two_products && forced == kSingle256) forced = kSingle128;
    if (forced >= 0 && (forced != kPair256 || pair_clusters > 0)) set_variant(pl, forced);
    else set_variant(pl, (pair_clusters > 0 && tiles * (tiles + 1) / 2 * 2 >= pair_clusters) ? kPair256 : single);
    pl.tiles_m = ceil_div(n, pl.tile_m);
    pl.tiles_n = ceil_div(n, pl.bn);
    pl.num_tiles = syrk_tile_count(mode, pl.tiles_m, pl.tiles_n, pl.tile_m, pl.bn);
    pl.full_tiles = pl.num_tiles;
    pl.kb_total = static_cast<int>(ceil_div(std::max<int64_t>(k, 1), bm::TILE_K)) * (two_products ? 2 : 1);
    pl.kb_per_split = pl.kb_total;
    const int64_t slots = pl.pair == 2 ? pair_clusters : sms;
    if (slots > 0 && pl.kb_total >= 8) {
        if (pl.num_tiles * 2 <= slots) {
            // (the same cap as GEMM: SYRK 512 x 8192 split 26 ways ran 23.3 us, 13 ways 14.3 us)
            try_split(pl, pl.num_tiles, std::min(kMaxAllSplits, ceil_div(slots, pl.num_tiles)), ws_bytes,
                      kSplitMinGainUs);
        } else {
            const int64_t tail = pl.num_tiles % slots;
            if (tail > 0 && tail * 2 <= slots)
                try_split(pl, tail, slots / tail, std::min(ws_bytes, kTailSplitMaxBytes), kSplitMinGainUs);
        }
    }
    size_grid(pl, sms, pair_clusters);
    return pl;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Tensor maps of one launch: operands, C, partial slots, MXFP8 scale atoms.
struct Maps {
    CUtensorMap a, b, c, p, sa, sb;
};

template <int ELEM, int EPI = bm::EPI_FULL>
cudaError_t launch_main(const cudaLaunchConfig_t &cfg, int variant, const Maps &t, const bm::GemmParams &prm)
{
    if constexpr (ELEM == bm::ELEM_MXF8) {
        if (variant == kSingle128Mx)
            return cudaLaunchKernelEx(&cfg, bm::bm_gemm_tcgen05_kernel<128, 5, 1, ELEM, 1, EPI>, t.a, t.b, t.c, t.p,
                                      t.sa, t.sb, prm);
        if (variant == kPair256Mx)
            return cudaLaunchKernelEx(&cfg, bm::bm_gemm_tcgen05_kernel<256, 5, 2, ELEM, 1, EPI>, t.a, t.b, t.c, t.p,
                                      t.sa, t.sb, prm);
        return cudaLaunchKernelEx(&cfg, bm::bm_gemm_tcgen05_kernel<128, 3, 2, ELEM, 2, EPI>, t.a, t.b, t.c, t.p, t.sa,
                                  t.sb, prm);
    } else {
        switch (variant) {
        case kSingle256:
            return cudaLaunchKernelEx(&cfg, bm::bm_gemm_tcgen05_kernel<256, 4, 1, ELEM, 1, EPI>, t.a, t.b, t.c, t.p,
                                      t.sa, t.sb, prm);
        case kSingle128:
            return cudaLaunchKernelEx(&cfg, bm::bm_gemm_tcgen05_kernel<128, 3, 1, ELEM, 2, EPI>, t.a, t.b, t.c, t.p,
                                      t.sa, t.sb, prm);
        default:
            return cudaLaunchKernelEx(&cfg, bm::bm_gemm_tcgen05_kernel<256, 3, 2, ELEM, 2, EPI>, t.a, t.b, t.c, t.p,
                                      t.sa, t.sb, prm);
        }
    }
}

// sa, sb: the MXFP8 scale maps (elem == ELEM_MXF8 only).
bm_status launch(const Plan &pl, const CUtensorMap &ta, const CUtensorMap &tb, bm::GemmParams &prm,
                 cudaStream_t stream, int sms, int elem = bm::ELEM_BF16, const CUtensorMap *sa = nullptr,
                 const CUtensorMap *sb = nullptr)
{
    // The epilogue moves C with TMA copies through a swizzled map (GEMM tiles, and
    // SYRK tiles inside the triangle). C is not prefetched into L2 ahead of the
    // epilogue: a prefetch copy occupies the same TMA unit as the operand copies
    // and cost more mainloop time than the load latency it hid.
    CUtensorMap tc;
    std::memset(&tc, 0, sizeof(tc));
    prm.tma_c = 0;
    const bm_ctype ct = prm.c_bf16 ? BM_C_BF16 : BM_C_F32;
    if (encode_c_tile(&tc, prm.C, ct, prm.m, prm.n, prm.ldc, prm.beta != 0.0f ? bm::CTA_M : 32u)) prm.tma_c = 1;
    // Half units place their columns in the TMA-store and group epilogues only: a call
    // whose C cannot take a tensor map runs its tail tiles whole.
    if (prm.n_split > 1 && !prm.tma_c) {
        prm.n_split = 1;
        prm.full_tiles = prm.num_tiles;
        prm.num_units = prm.num_tiles;
    }
    CUtensorMap tp;
    std::memset(&tp, 0, sizeof(tp));
    prm.store_p_tma = 0;
    if (prm.k_splits > 1 && prm.partial != nullptr &&
        encode_slots(&tp, prm.partial, (prm.num_tiles - prm.full_tiles) * prm.k_splits * pl.tile_m, pl.bn))
        prm.store_p_tma = 1;
    prm.fixup = 0;
    if (pl.fixup && prm.k_splits > 1 && prm.partial != nullptr) {
        static std::atomic<unsigned long long> seq{0};
        prm.fixup = 1;
        prm.fixup_ctr = reinterpret_cast<unsigned long long *>(reinterpret_cast<char *>(prm.partial) + pl.slot_bytes);
        prm.seq = (seq.fetch_add(1) % ((1ull << 48) - 1)) + 1;  // 1 .. 2^48 - 1
    }
    if (pl.ctas <= 0) return BM_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    cfg.gridDim = dim3(static_cast<unsigned>(pl.ctas), 1, 1);
    cfg.blockDim = dim3(bm::NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(variant_smem(pl.variant));
    cfg.stream = stream;
    cfg.attrs = attr;
    // programmatic dependent launch: the kernel's set-up may overlap the previous kernel's tail
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 1;
    if (pl.pair == 2) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = 2;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    // A GEMM runs a kernel copy without the SYRK diagonal path: TMA-store epilogue
    // for beta == 0, group combine otherwise (split units as in the full kernel;
    // for E4M3 only the beta == 0 copy exists).
    const bool lean = prm.mode == bm::MODE_GEMM && prm.tma_c;
    cudaError_t err;
    Maps t;
    std::memset(&t, 0, sizeof(t));
    t.a = ta;
    t.b = tb;
    t.c = tc;
    t.p = tp;
    if (sa != nullptr) t.sa = *sa;
    if (sb != nullptr) t.sb = *sb;
    if (elem == bm::ELEM_MXF8 && (sa == nullptr || sb == nullptr)) return BM_ERR_CUDA;
    if (elem == bm::ELEM_MXF8 && lean && prm.beta == 0.0f)
        err = launch_main<bm::ELEM_MXF8, bm::EPI_STORE>(cfg, pl.variant, t, prm);
    else if (elem == bm::ELEM_MXF8) err = launch_main<bm::ELEM_MXF8>(cfg, pl.variant, t, prm);
    else if (elem == bm::ELEM_E4M3 && lean && prm.beta == 0.0f)
        err = launch_main<bm::ELEM_E4M3, bm::EPI_STORE>(cfg, pl.variant, t, prm);
    else if (elem == bm::ELEM_E4M3) err = launch_main<bm::ELEM_E4M3>(cfg, pl.variant, t, prm);
    else if (lean && prm.beta == 0.0f) err = launch_main<bm::ELEM_BF16, bm::EPI_STORE>(cfg, pl.variant, t, prm);
    else if (lean) err = launch_main<bm::ELEM_BF16, bm::EPI_COMBINE>(cfg, pl.variant, t, prm);
    else err = launch_main<bm::ELEM_BF16>(cfg, pl.variant, t, prm);
    if (err != cudaSuccess) {
        cudaGetLastError();
        return BM_ERR_CUDA;
    }
    if (prm.k_splits > 1 && !prm.fixup) {
        const int64_t work = (prm.num_tiles - prm.full_tiles) * pl.tile_m * (pl.bn / 4);
        const int blocks =
            static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(ceil_div(work, 256), 8 * static_cast<int64_t>(sms))));
        cudaLaunchConfig_t rc = {};
        cudaLaunchAttribute ra[1];
        ra[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        ra[0].val.programmaticStreamSerializationAllowed = 1;
        rc.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
        rc.blockDim = dim3(256, 1, 1);
        rc.stream = stream;
        rc.attrs = ra;
        rc.numAttrs = 1;
        cudaError_t re;
        switch (pl.variant) {
        case kSingle256: re = cudaLaunchKernelEx(&rc, bm::bm_splitk_reduce_kernel<128, 256>, prm); break;
        case kSingle128:
        case kSingle128Mx: re = cudaLaunchKernelEx(&rc, bm::bm_splitk_reduce_kernel<128, 128>, prm); break;
        case kPair128Mx: re = cudaLaunchKernelEx(&rc, bm::bm_splitk_reduce_kernel<256, 128>, prm); break;
        case kPair256Mx: re = cudaLaunchKernelEx(&rc, bm::bm_splitk_reduce_kernel<256, 256>, prm); break;
        default: re = cudaLaunchKernelEx(&rc, bm::bm_splitk_reduce_kernel<256, 256>, prm); break;
        }
        if (re != cudaSuccess) {
            cudaGetLastError();
            return BM_ERR_CUDA;
        }
        if (cudaGetLastError() != cudaSuccess) return BM_ERR_CUDA;
    }
    return BM_OK;
}

// C = beta * C (alpha == 0 or k == 0): a grid-stride kernel of at most 8 blocks per SM.
bm_status launch_scale(bm::GemmParams &prm, cudaStream_t stream, int sms)
{
    const int64_t work = prm.m * ceil_div(prm.n, 4);
    const int blocks =
        static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(ceil_div(work, 256), 8 * static_cast<int64_t>(sms))));
    cudaLaunchConfig_t rc = {};
    cudaLaunchAttribute ra[1];
    ra[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    ra[0].val.programmaticStreamSerializationAllowed = 1;
    rc.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
    rc.blockDim = dim3(256, 1, 1);
    rc.stream = stream;
    rc.attrs = ra;
    rc.numAttrs = 1;
    if (cudaLaunchKernelEx(&rc, bm::bm_scale_kernel, prm) != cudaSuccess) {
        cudaGetLastError();
        return BM_ERR_CUDA;
    }
    return BM_OK;
}

void fill_params(bm::GemmParams &prm, const Plan &pl)
{
    prm.tiles_m = pl.tiles_m;
    prm.tiles_n = pl.tiles_n;
    prm.num_tiles = pl.num_tiles;
    prm.full_tiles = pl.full_tiles;
    prm.num_units = pl.num_units;
    prm.k_splits = pl.k_splits;
    prm.n_split = pl.n_split;
    prm.kb_per_split = pl.kb_per_split;
    prm.kb_total = pl.kb_total;
}

void export_plan(const Plan &pl, bm_plan *plan)
{
    plan->tile_m = pl.tile_m;
    plan->tile_n = pl.bn;
    plan->tile_k = bm::TILE_K;
    plan->stages = pl.stages;
    plan->tiles = pl.num_tiles;
    plan->k_splits = pl.k_splits;
    plan->split_tiles = pl.num_tiles - pl.full_tiles;
    plan->ctas = pl.ctas;
    plan->cta_pair = pl.pair;
    plan->kernels = pl.k_splits > 1 && !pl.fixup ? 2 : 1;
    plan->workspace_bytes = pl.k_splits > 1 ? pl.ws_bytes : 0;
    plan->stage_kblocks = kVariantStageKBlocks[pl.variant];
    plan->n_splits = pl.n_split;
}

// Pair-cluster capacity for planning without a device (host-only planning): one per SM pair.
int pair_clusters_or_default(int sms, bool mxfp8 = false)
{
    int dev = -1;
    if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < kMaxDevices) {
        std::lock_guard<std::mutex> lock(g_mutex);
        if (g_devices[dev].attrs_set)
            return mxfp8 ? g_devices[dev].max_pair_clusters_mx : g_devices[dev].max_pair_clusters;
    }
    cudaGetLastError();
    return sms / 2;
}

bm::GemmParams base_params(int64_t m, int64_t n, int64_t k, float alpha, float beta, void *C, int64_t ldc,
                           bm_ctype ct, DeviceState *st)
{
    bm::GemmParams p;
    std::memset(&p, 0, sizeof(p));
    p.m = m;
    p.n = n;
    p.k = k;
    p.C = C;
    p.ldc = ldc;
    p.alpha = alpha;
    p.beta = beta;
    p.c_bf16 = ct == BM_C_BF16 ? 1 : 0;
    p.k_splits = 1;
    p.group_m = kGroupM;
    p.status = st != nullptr ? st->status : nullptr;
    p.timeout_ns = static_cast<uint64_t>(g_timeout_ms.load()) * 1000000ull;
    p.debug_stall = g_debug_stall.load();
    return p;
}

bm_status check_gemm_args(int64_t m, int64_t n, int64_t k, int transA, int transB, int64_t lda, int64_t ldb,
                          int64_t ldc, int ct)
{
    if (m < 0 || n < 0 || k < 0) return BM_ERR_INVALID_VALUE;
    if (!fits_int32(m) || !fits_int32(n) || !fits_int32(k)) return BM_ERR_INVALID_VALUE;
    if ((transA != BM_OP_N && transA != BM_OP_T) || (transB != BM_OP_N && transB != BM_OP_T))
        return BM_ERR_INVALID_VALUE;
    if (ct != BM_C_F32 && ct != BM_C_BF16) return BM_ERR_INVALID_VALUE;
    const int64_t need_a = transA == BM_OP_N ? k : m;
    const int64_t need_b = transB == BM_OP_N ? n : k;
    if (lda < std::max<int64_t>(1, need_a) || ldb < std::max<int64_t>(1, need_b) || ldc < std::max<int64_t>(1, n))
        return BM_ERR_INVALID_VALUE;
    return BM_OK;
}

// ---------------------------------------------------------------- allocation-free GEMM
// Scratch for bm_gemm_bf16_noalloc: the split-K partials live in this file-scope
// device array instead of a caller or library allocation. Every GPU that loads
// the library holds it until the process exits. In host code the symbol is only
// a host-side stand-in; the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) float g_noalloc_scratch[BM_NOALLOC_SCRATCH_BYTES / sizeof(float)];

float *g_noalloc_scratch_addr[kMaxDevices] = {};

// Set-up for the allocation-free entry point on the current device: the device
// checks and one-time attributes of the other entry points without any
// allocation, plus the device address of the scratch array, looked up once per
// device with that device current.
bm_status noalloc_device_setup(DeviceState **out, float **scratch)
{
    DeviceState *st = nullptr;
    const bm_status s = device_state(&st, false);
    if (s != BM_OK) return s;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_noalloc_scratch_addr[st->device] == nullptr) {
        void *addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || addr == nullptr) {
            cudaGetLastError();
            return BM_ERR_CUDA;
        }
        g_noalloc_scratch_addr[st->device] = static_cast<float *>(addr);
    }
    *scratch = g_noalloc_scratch_addr[st->device];
    *out = st;
    return BM_OK;
}

}  // namespace

extern "C" {

bm_status bm_gemm_bf16(int64_t m, int64_t n, int64_t k, bm_op transA, bm_op transB, float alpha, const void *A,
                       int64_t lda, const void *B, int64_t ldb, float beta, void *C, int64_t ldc, bm_ctype c_type,
                       void *workspace, size_t workspace_bytes, bm_stream_t stream)
{
    bm_status s = check_gemm_args(m, n, k, transA, transB, lda, ldb, ldc, c_type);
    if (s != BM_OK) return s;
    if (workspace_bytes > 0 && (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0))
        return BM_ERR_WORKSPACE;
    if (m == 0 || n == 0) return BM_OK;
    const bool products = alpha != 0.0f && k > 0;
    if (C == nullptr || (products && (A == nullptr || B == nullptr))) return BM_ERR_INVALID_VALUE;
    const int64_t esz = c_type == BM_C_BF16 ? 2 : 4;
    if (!aligned16(C) || (ldc * esz) % 16 != 0) return BM_ERR_MISALIGNED;
    if (products && (!aligned16(A) || !aligned16(B) || (lda * 2) % 16 != 0 || (ldb * 2) % 16 != 0))
        return BM_ERR_MISALIGNED;
    DeviceState *st = nullptr;
    s = device_state(&st);
    if (s != BM_OK) return s;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    bm::GemmParams prm = base_params(m, n, k, alpha, beta, C, ldc, c_type, st);
    prm.mode = bm::MODE_GEMM;
    if (!products) return launch_scale(prm, cs, st->sm_count);

    const Plan pl = plan_gemm(m, n, k, workspace != nullptr ? workspace_bytes : 0, st->sm_count,
                              st->max_pair_clusters, bm::ELEM_BF16, beta != 0.0f);
    CUtensorMap ta, tb;
    const bool a_mn = transA == BM_OP_T, b_mn = transB == BM_OP_N;
    // each CTA stages 128 rows of op(A) and bn / pair rows of op(B)^T
    if (!encode_operand(&ta, A, a_mn, m, k, lda, bm::CTA_M)) return BM_ERR_CUDA;
    if (!encode_operand(&tb, B, b_mn, n, k, ldb, static_cast<uint32_t>(pl.bn / pl.pair))) return BM_ERR_CUDA;
    prm.a_mn_major = a_mn;
    prm.b_mn_major = b_mn;
    const int kps = kVariantStageKBlocks[pl.variant];
    prm.a_box3 = encode_stage_box(&ta, A, bm::ELEM_BF16, a_mn, m, k, lda, bm::CTA_M, kps);
    prm.b_box3 = encode_stage_box(&tb, B, bm::ELEM_BF16, b_mn, n, k, ldb, pl.bn / pl.pair, kps);
    fill_params(prm, pl);
    prm.partial = pl.k_splits > 1 ? static_cast<float *>(workspace) : nullptr;
    return launch(pl, ta, tb, prm, cs, st->sm_count);
}

size_t bm_gemm_bf16_workspace_size(int64_t m, int64_t n, int64_t k)
{
    if (m <= 0 || n <= 0 || k <= 0) return 0;
    const int sms = sm_count_or_default();
    const Plan pl = plan_gemm(m, n, k, SIZE_MAX, sms, pair_clusters_or_default(sms));
    return pl.k_splits > 1 ? pl.ws_bytes : 0;
}

bm_status bm_gemm_bf16_noalloc(int64_t m, int64_t n, int64_t k, bm_op transA, bm_op transB, float alpha,
                               const void *A, int64_t lda, const void *B, int64_t ldb, float beta, void *C,
                               int64_t ldc, bm_ctype c_type, bm_stream_t stream)
{
    bm_status s = check_gemm_args(m, n, k, transA, transB, lda, ldb, ldc, c_type);
    if (s != BM_OK) return s;
    if (m == 0 || n == 0) return BM_OK;
    const bool products = alpha != 0.0f && k > 0;
    if (C == nullptr || (products && (A == nullptr || B == nullptr))) return BM_ERR_INVALID_VALUE;
    const int64_t esz = c_type == BM_C_BF16 ? 2 : 4;
    if (!aligned16(C) || (ldc * esz) % 16 != 0) return BM_ERR_MISALIGNED;
    if (products && (!aligned16(A) || !aligned16(B) || (lda * 2) % 16 != 0 || (ldb * 2) % 16 != 0))
        return BM_ERR_MISALIGNED;
    DeviceState *st = nullptr;
    float *scratch = nullptr;
    s = noalloc_device_setup(&st, &scratch);
    if (s != BM_OK) return s;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    bm::GemmParams prm = base_params(m, n, k, alpha, beta, C, ldc, c_type, st);
    prm.mode = bm::MODE_GEMM;
    if (!products) return launch_scale(prm, cs, st->sm_count);

    // The plan bm_gemm_bf16 makes with a workspace the size of the static array:
    // the planner lowers the split count until the partials fit.
    const Plan pl = plan_gemm(m, n, k, BM_NOALLOC_SCRATCH_BYTES, st->sm_count, st->max_pair_clusters,
                              bm::ELEM_BF16, beta != 0.0f);
    if (pl.k_splits > 1 && pl.ws_bytes > BM_NOALLOC_SCRATCH_BYTES) return BM_ERR_WORKSPACE;  // defensive
    CUtensorMap ta, tb;
    const bool a_mn = transA == BM_OP_T, b_mn = transB == BM_OP_N;
    if (!encode_operand(&ta, A, a_mn, m, k, lda, bm::CTA_M)) return BM_ERR_CUDA;
    if (!encode_operand(&tb, B, b_mn, n, k, ldb, static_cast<uint32_t>(pl.bn / pl.pair))) return BM_ERR_CUDA;
    prm.a_mn_major = a_mn;
    prm.b_mn_major = b_mn;
    const int kps = kVariantStageKBlocks[pl.variant];
    prm.a_box3 = encode_stage_box(&ta, A, bm::ELEM_BF16, a_mn, m, k, lda, bm::CTA_M, kps);
    prm.b_box3 = encode_stage_box(&tb, B, bm::ELEM_BF16, b_mn, n, k, ldb, pl.bn / pl.pair, kps);
    fill_params(prm, pl);
    prm.partial = pl.k_splits > 1 ? scratch : nullptr;
    return launch(pl, ta, tb, prm, cs, st->sm_count);
}

bm_status bm_syrk_bf16(bm_uplo uplo, bm_op trans, int64_t n, int64_t k, float alpha, const void *A, int64_t lda,
                       float beta, void *C, int64_t ldc, bm_ctype c_type, void *workspace, size_t workspace_bytes,
                       bm_stream_t stream)
{
    if (uplo != BM_LOWER && uplo != BM_UPPER) return BM_ERR_INVALID_VALUE;
    if (n < 0 || k < 0 || !fits_int32(n) || !fits_int32(k)) return BM_ERR_INVALID_VALUE;
    if (trans != BM_OP_N && trans != BM_OP_T) return BM_ERR_INVALID_VALUE;
    if (c_type != BM_C_F32 && c_type != BM_C_BF16) return BM_ERR_INVALID_VALUE;
    const int64_t need_a = trans == BM_OP_N ? k : n;
    if (lda < std::max<int64_t>(1, need_a) || ldc < std::max<int64_t>(1, n)) return BM_ERR_INVALID_VALUE;
    if (workspace_bytes > 0 && (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0))
        return BM_ERR_WORKSPACE;
    if (n == 0) return BM_OK;
    const bool products = alpha != 0.0f && k > 0;
    if (C == nullptr || (products && A == nullptr)) return BM_ERR_INVALID_VALUE;
    const int64_t esz = c_type == BM_C_BF16 ? 2 : 4;
    if (!aligned16(C) || (ldc * esz) % 16 != 0) return BM_ERR_MISALIGNED;
    if (products && (!aligned16(A) || (lda * 2) % 16 != 0)) return BM_ERR_MISALIGNED;
    DeviceState *st = nullptr;
    bm_status s = device_state(&st);
    if (s != BM_OK) return s;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    bm::GemmParams prm = base_params(n, n, k, alpha, beta, C, ldc, c_type, st);
    prm.mode = uplo == BM_LOWER ? bm::MODE_SYRK_LOWER : bm::MODE_SYRK_UPPER;
    if (!products) return launch_scale(prm, cs, st->sm_count);

    const Plan pl = plan_syrk(prm.mode, n, k, workspace != nullptr ? workspace_bytes : 0, st->sm_count,
                              st->max_pair_clusters);
    CUtensorMap ta, tb;
    const bool mn = trans == BM_OP_T;  // A stored [k][n]: both operands are M/N-major
    if (!encode_operand(&ta, A, mn, n, k, lda, bm::CTA_M)) return BM_ERR_CUDA;
    if (!encode_operand(&tb, A, mn, n, k, lda, static_cast<uint32_t>(pl.bn / pl.pair))) return BM_ERR_CUDA;
    prm.a_mn_major = mn;
    prm.b_mn_major = mn;
    const int kps = kVariantStageKBlocks[pl.variant];
    prm.a_box3 = encode_stage_box(&ta, A, bm::ELEM_BF16, mn, n, k, lda, bm::CTA_M, kps);
    prm.b_box3 = encode_stage_box(&tb, A, bm::ELEM_BF16, mn, n, k, lda, pl.bn / pl.pair, kps);
    fill_params(prm, pl);
    prm.partial = pl.k_splits > 1 ? static_cast<float *>(workspace) : nullptr;
    return launch(pl, ta, tb, prm, cs, st->sm_count);
}

bm_status bm_syr2k_bf16(bm_uplo uplo, bm_op trans, int64_t n, int64_t k, float alpha, const void *A, int64_t lda,
                        const void *B, int64_t ldb, float beta, void *C, int64_t ldc, bm_ctype c_type,
                        void *workspace, size_t workspace_bytes, bm_stream_t stream)
{
    if (uplo != BM_LOWER && uplo != BM_UPPER) return BM_ERR_INVALID_VALUE;
    if (n < 0 || k < 0 || !fits_int32(n) || !fits_int32(k)) return BM_ERR_INVALID_VALUE;
    if (trans != BM_OP_N && trans != BM_OP_T) return BM_ERR_INVALID_VALUE;
    if (c_type != BM_C_F32 && c_type != BM_C_BF16) return BM_ERR_INVALID_VALUE;
    const int64_t need = trans == BM_OP_N ? k : n;
    if (lda < std::max<int64_t>(1, need) || ldb < std::max<int64_t>(1, need) || ldc < std::max<int64_t>(1, n))
        return BM_ERR_INVALID_VALUE;
    if (workspace_bytes > 0 && (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0))
        return BM_ERR_WORKSPACE;
    if (n == 0) return BM_OK;
    const bool products = alpha != 0.0f && k > 0;
    if (C == nullptr || (products && (A == nullptr || B == nullptr))) return BM_ERR_INVALID_VALUE;
    const int64_t esz = c_type == BM_C_BF16 ? 2 : 4;
    if (!aligned16(C) || (ldc * esz) % 16 != 0) return BM_ERR_MISALIGNED;
    if (products && (!aligned16(A) || !aligned16(B) || (lda * 2) % 16 != 0 || (ldb * 2) % 16 != 0))
        return BM_ERR_MISALIGNED;
    DeviceState *st = nullptr;
    bm_status s = device_state(&st);
    if (s != BM_OK) return s;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    bm::GemmParams prm = base_params(n, n, k, alpha, beta, C, ldc, c_type, st);
    prm.mode = uplo == BM_LOWER ? bm::MODE_SYRK_LOWER : bm::MODE_SYRK_UPPER;
    if (!products) return launch_scale(prm, cs, st->sm_count);

    const Plan pl = plan_syrk(prm.mode, n, k, workspace != nullptr ? workspace_bytes : 0, st->sm_count,
                              st->max_pair_clusters, true);
    CUtensorMap ta, tb;
    const bool mn = trans == BM_OP_T;  // A, B stored [k][n]: both operands are M/N-major
    // Both maps serve as the A operand (128 rows) and the B operand (bn / pair = 128 rows).
    if (!encode_operand(&ta, A, mn, n, k, lda, bm::CTA_M)) return BM_ERR_CUDA;
    if (!encode_operand(&tb, B, mn, n, k, ldb, bm::CTA_M)) return BM_ERR_CUDA;
    prm.a_mn_major = mn;
    prm.b_mn_major = mn;
    fill_params(prm, pl);
    prm.syr2k_kb = pl.kb_total / 2;
    prm.partial = pl.k_splits > 1 ? static_cast<float *>(workspace) : nullptr;
    // Stage boxes when no stage straddles the swap of A and B (both maps then serve
    // as stage boxes of 128 rows in both roles): the swap on a stage boundary, and
    // no K split (a split may start a unit, and so its stages, at any k-block).
    const int kps = kVariantStageKBlocks[pl.variant];
    if (prm.syr2k_kb % kps == 0 && pl.k_splits == 1) {
        CUtensorMap ta3 = ta, tb3 = tb;
        if (encode_stage_box(&ta3, A, bm::ELEM_BF16, mn, n, k, lda, bm::CTA_M, kps) &&
            encode_stage_box(&tb3, B, bm::ELEM_BF16, mn, n, k, ldb, bm::CTA_M, kps)) {
            ta = ta3;
            tb = tb3;
            prm.a_box3 = 1;
            prm.b_box3 = 1;
        }
    }
    return launch(pl, ta, tb, prm, cs, st->sm_count);
}

bm_status bm_gemm_e4m3(int64_t m, int64_t n, int64_t k, float alpha, const void *A, int64_t lda, const void *B,
                       int64_t ldb, float beta, void *C, int64_t ldc, bm_ctype c_type, void *workspace,
                       size_t workspace_bytes, bm_stream_t stream)
{
    // A [m, k] and B [n, k] row-major: both operands K-major (op(B) = B^T)
    bm_status s = check_gemm_args(m, n, k, BM_OP_N, BM_OP_T, lda, ldb, ldc, c_type);
    if (s != BM_OK) return s;
    if (workspace_bytes > 0 && (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0))
        return BM_ERR_WORKSPACE;
    if (m == 0 || n == 0) return BM_OK;
    const bool products = alpha != 0.0f && k > 0;
    if (C == nullptr || (products && (A == nullptr || B == nullptr))) return BM_ERR_INVALID_VALUE;
    const int64_t esz = c_type == BM_C_BF16 ? 2 : 4;
    if (!aligned16(C) || (ldc * esz) % 16 != 0) return BM_ERR_MISALIGNED;
    if (products && (!aligned16(A) || !aligned16(B) || lda % 16 != 0 || ldb % 16 != 0)) return BM_ERR_MISALIGNED;
    DeviceState *st = nullptr;
    s = device_state(&st);
    if (s != BM_OK) return s;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    bm::GemmParams prm = base_params(m, n, k, alpha, beta, C, ldc, c_type, st);
    prm.mode = bm::MODE_GEMM;
    if (!products) return launch_scale(prm, cs, st->sm_count);

    const Plan pl = plan_gemm(m, n, k, workspace != nullptr ? workspace_bytes : 0, st->sm_count,
                              st->max_pair_clusters, bm::ELEM_E4M3);
    CUtensorMap ta, tb;
    const uint32_t kb = static_cast<uint32_t>(bm::kblock_elems(bm::ELEM_E4M3));
    if (!encode_operand_2d(&ta, A, bm::ELEM_E4M3, k, m, lda, kb, bm::CTA_M)) return BM_ERR_CUDA;
    if (!encode_operand_2d(&tb, B, bm::ELEM_E4M3, k, n, ldb, kb, static_cast<uint32_t>(pl.bn / pl.pair)))
        return BM_ERR_CUDA;
    prm.a_mn_major = 0;
    prm.b_mn_major = 0;
    const int kps = kVariantStageKBlocks[pl.variant];
    prm.a_box3 = encode_stage_box(&ta, A, bm::ELEM_E4M3, false, m, k, lda, bm::CTA_M, kps);
    prm.b_box3 = encode_stage_box(&tb, B, bm::ELEM_E4M3, false, n, k, ldb, pl.bn / pl.pair, kps);
    fill_params(prm, pl);
    prm.partial = pl.k_splits > 1 ? static_cast<float *>(workspace) : nullptr;
    return launch(pl, ta, tb, prm, cs, st->sm_count, bm::ELEM_E4M3);
}

size_t bm_gemm_e4m3_workspace_size(int64_t m, int64_t n, int64_t k)
{
    if (m <= 0 || n <= 0 || k <= 0) return 0;
    const int sms = sm_count_or_default();
    const Plan pl = plan_gemm(m, n, k, SIZE_MAX, sms, pair_clusters_or_default(sms), bm::ELEM_E4M3);
    return pl.k_splits > 1 ? pl.ws_bytes : 0;
}

bm_status bm_gemm_mxfp8(int64_t m, int64_t n, int64_t k, float alpha, const void *A, int64_t lda, const void *SFA,
                        const void *B, int64_t ldb, const void *SFB, float beta, void *C, int64_t ldc,
                        bm_ctype c_type, void *workspace, size_t workspace_bytes, bm_stream_t stream)
{
    // A [m, k] and B [n, k] row-major E4M3 codes (both operands K-major), scale atoms beside them
    bm_status s = check_gemm_args(m, n, k, BM_OP_N, BM_OP_T, lda, ldb, ldc, c_type);
    if (s != BM_OK) return s;
    if (workspace_bytes > 0 && (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0))
        return BM_ERR_WORKSPACE;
    if (m == 0 || n == 0) return BM_OK;
    const bool products = alpha != 0.0f && k > 0;
    if (C == nullptr || (products && (A == nullptr || B == nullptr || SFA == nullptr || SFB == nullptr)))
        return BM_ERR_INVALID_VALUE;
    const int64_t esz = c_type == BM_C_BF16 ? 2 : 4;
    if (!aligned16(C) || (ldc * esz) % 16 != 0) return BM_ERR_MISALIGNED;
    if (products && (!aligned16(A) || !aligned16(B) || !aligned16(SFA) || !aligned16(SFB) || lda % 16 != 0 ||
                     ldb % 16 != 0))
        return BM_ERR_MISALIGNED;
    DeviceState *st = nullptr;
    s = device_state(&st);
    if (s != BM_OK) return s;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    bm::GemmParams prm = base_params(m, n, k, alpha, beta, C, ldc, c_type, st);
    prm.mode = bm::MODE_GEMM;
    if (!products) return launch_scale(prm, cs, st->sm_count);

    const Plan pl = plan_gemm(m, n, k, workspace != nullptr ? workspace_bytes : 0, st->sm_count,
                              st->max_pair_clusters_mx, bm::ELEM_MXF8);
    CUtensorMap ta, tb, tsa, tsb;
    const uint32_t kb = static_cast<uint32_t>(bm::kblock_elems(bm::ELEM_E4M3));
    if (!encode_operand_2d(&ta, A, bm::ELEM_E4M3, k, m, lda, kb, bm::CTA_M)) return BM_ERR_CUDA;
    if (!encode_operand_2d(&tb, B, bm::ELEM_E4M3, k, n, ldb, kb, static_cast<uint32_t>(pl.bn / pl.pair)))
        return BM_ERR_CUDA;
    const int kps = kVariantStageKBlocks[pl.variant];
    // each CTA takes the A scales of its 128 rows and the B scales of all the tile's columns
    if (!encode_scales(&tsa, SFA, m, k, kps, 1)) return BM_ERR_CUDA;
    if (!encode_scales(&tsb, SFB, n, k, kps, pl.bn / 128)) return BM_ERR_CUDA;
    prm.a_mn_major = 0;
    prm.b_mn_major = 0;
    prm.a_box3 = encode_stage_box(&ta, A, bm::ELEM_E4M3, false, m, k, lda, bm::CTA_M, kps);
    prm.b_box3 = encode_stage_box(&tb, B, bm::ELEM_E4M3, false, n, k, ldb, pl.bn / pl.pair, kps);
    fill_params(prm, pl);
    prm.partial = pl.k_splits > 1 ? static_cast<float *>(workspace) : nullptr;
    return launch(pl, ta, tb, prm, cs, st->sm_count, bm::ELEM_MXF8, &tsa, &tsb);
}

size_t bm_gemm_mxfp8_workspace_size(int64_t m, int64_t n, int64_t k)
{
    if (m <= 0 || n <= 0 || k <= 0) return 0;
    const int sms = sm_count_or_default();
    const Plan pl = plan_gemm(m, n, k, SIZE_MAX, sms, pair_clusters_or_default(sms, true), bm::ELEM_MXF8);
    return pl.k_splits > 1 ? pl.ws_bytes : 0;
}

bm_status bm_quantize_mxfp8(int64_t rows, int64_t k, const void *X, int64_t ldx, void *Q, int64_t ldq, void *S,
                            bm_stream_t stream)
{
    if (rows < 0 || k < 0 || !fits_int32(rows) || !fits_int32(k)) return BM_ERR_INVALID_VALUE;
    if (ldx < std::max<int64_t>(1, k) || ldq < std::max<int64_t>(1, k)) return BM_ERR_INVALID_VALUE;
    if (rows == 0 || k == 0) return BM_OK;
    if (X == nullptr || Q == nullptr || S == nullptr) return BM_ERR_INVALID_VALUE;
    if (!aligned16(X) || !aligned16(Q) || !aligned16(S) || (ldx * 2) % 16 != 0 || ldq % 16 != 0)
        return BM_ERR_MISALIGNED;
    DeviceState *st = nullptr;
    const bm_status s = device_state(&st);
    if (s != BM_OK) return s;
    bm::QuantParams p;
    p.rows = rows;
    p.k = k;
    p.X = static_cast<const uint16_t *>(X);
    p.ldx = ldx;
    p.Q = static_cast<uint8_t *>(Q);
    p.ldq = ldq;
    p.S = static_cast<uint8_t *>(S);
    p.groups = ceil_div(k, 32);
    p.groups_pad = 4 * ceil_div(k, 128);
    p.rows_pad = 128 * ceil_div(rows, 128);
    // One thread per group of 32; a grid-stride loop over at most 8 blocks of 256 per SM.
    // Four blocks fit on an SM at once, so that is two whole waves. Measured, against a
    // cap of 16 (4096^2: 2048 blocks, 3.4 waves): 4096^2 10.2 -> 9.6 us, 8192^2
    // 32.0 -> 31.4 us, 2048 x 4096 unchanged; a cap of 4 (one wave) was slower.
    const int64_t work = p.rows_pad * p.groups_pad;
    const int blocks =
        static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(ceil_div(work, 256), 8 * static_cast<int64_t>(st->sm_count))));
    cudaLaunchConfig_t rc = {};
    cudaLaunchAttribute ra[1];
    ra[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    ra[0].val.programmaticStreamSerializationAllowed = 1;
    rc.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
    rc.blockDim = dim3(256, 1, 1);
    rc.stream = reinterpret_cast<cudaStream_t>(stream);
    rc.attrs = ra;
    rc.numAttrs = 1;
    if (cudaLaunchKernelEx(&rc, bm::bm_quantize_mxfp8_kernel, p) != cudaSuccess) {
        cudaGetLastError();
        return BM_ERR_CUDA;
    }
    return BM_OK;
}

bm_status bm_gemm_mxfp8_plan(int64_t m, int64_t n, int64_t k, size_t workspace_bytes, bm_plan *plan)
{
    if (plan == nullptr) return BM_ERR_INVALID_VALUE;
    if (m < 0 || n < 0 || k < 0 || !fits_int32(m) || !fits_int32(n) || !fits_int32(k)) return BM_ERR_INVALID_VALUE;
    std::memset(plan, 0, sizeof(*plan));
    if (m == 0 || n == 0) return BM_OK;
    if (k == 0) {
        plan->kernels = 1;
        return BM_OK;
    }
    const int sms = sm_count_or_default();
    export_plan(plan_gemm(m, n, k, workspace_bytes, sms, pair_clusters_or_default(sms, true), bm::ELEM_MXF8), plan);
    plan->tile_k = 128;
    return BM_OK;
}

bm_status bm_gemm_bf16_plan(int64_t m, int64_t n, int64_t k, size_t workspace_bytes, bm_plan *plan)
{
    if (plan == nullptr) return BM_ERR_INVALID_VALUE;
    if (m < 0 || n < 0 || k < 0 || !fits_int32(m) || !fits_int32(n) || !fits_int32(k)) return BM_ERR_INVALID_VALUE;
    std::memset(plan, 0, sizeof(*plan));
    if (m == 0 || n == 0) return BM_OK;
    if (k == 0) {
        plan->kernels = 1;
        return BM_OK;
    }
    const int sms = sm_count_or_default();
    export_plan(plan_gemm(m, n, k, workspace_bytes, sms, pair_clusters_or_default(sms)), plan);
    return BM_OK;
}

bm_status bm_syrk_bf16_plan(bm_uplo uplo, int64_t n, int64_t k, size_t workspace_bytes, bm_plan *plan)
{
    if (plan == nullptr || (uplo != BM_LOWER && uplo != BM_UPPER)) return BM_ERR_INVALID_VALUE;
    if (n < 0 || k < 0 || !fits_int32(n) || !fits_int32(k)) return BM_ERR_INVALID_VALUE;
    std::memset(plan, 0, sizeof(*plan));
    if (n == 0) return BM_OK;
    if (k == 0) {
        plan->kernels = 1;
        return BM_OK;
    }
    const int sms = sm_count_or_default();
    export_plan(plan_syrk(uplo == BM_LOWER ? bm::MODE_SYRK_LOWER : bm::MODE_SYRK_UPPER, n, k, workspace_bytes, sms,
                          pair_clusters_or_default(sms)),
                plan);
    return BM_OK;
}

size_t bm_syrk_bf16_workspace_size(bm_uplo uplo, int64_t n, int64_t k)
{
    if (n <= 0 || k <= 0 || (uplo != BM_LOWER && uplo != BM_UPPER)) return 0;
    const int sms = sm_count_or_default();
    const Plan pl = plan_syrk(uplo == BM_LOWER ? bm::MODE_SYRK_LOWER : bm::MODE_SYRK_UPPER, n, k, SIZE_MAX, sms,
                              pair_clusters_or_default(sms));
    return pl.k_splits > 1 ? pl.ws_bytes : 0;
}

size_t bm_syr2k_bf16_workspace_size(bm_uplo uplo, int64_t n, int64_t k)
{
    if (n <= 0 || k <= 0 || (uplo != BM_LOWER && uplo != BM_UPPER)) return 0;
    const int sms = sm_count_or_default();
    const Plan pl = plan_syrk(uplo == BM_LOWER ? bm::MODE_SYRK_LOWER : bm::MODE_SYRK_UPPER, n, k, SIZE_MAX, sms,
                              pair_clusters_or_default(sms), true);
    return pl.k_splits > 1 ? pl.ws_bytes : 0;
}

bm_status bm_syrk_bf16_tile_order(bm_uplo uplo, int64_t n, int64_t k, int64_t count, int64_t *tile_row,
                                   int64_t *tile_col)
{
    if (uplo != BM_LOWER && uplo != BM_UPPER) return BM_ERR_INVALID_VALUE;
    if (n < 0 || k < 0 || count < 0 || !fits_int32(n) || !fits_int32(k)) return BM_ERR_INVALID_VALUE;
    if (count > 0 && (tile_row == nullptr || tile_col == nullptr)) return BM_ERR_INVALID_VALUE;
    if (n == 0 || k == 0) return count == 0 ? BM_OK : BM_ERR_INVALID_VALUE;
    const int sms = sm_count_or_default();
    const int mode = uplo == BM_LOWER ? bm::MODE_SYRK_LOWER : bm::MODE_SYRK_UPPER;
    const Plan pl = plan_syrk(mode, n, k, 0, sms, pair_clusters_or_default(sms));
    if (count != pl.num_tiles) return BM_ERR_INVALID_VALUE;
    for (int64_t t = 0; t < count; ++t) syrk_coords(mode, pl.tiles_m, pl.tiles_n, pl.tile_m, pl.bn, t, tile_row[t], tile_col[t]);
    return BM_OK;
}

bm_status bm_get_last_device_error(bm_stream_t stream)
{
    DeviceState *st = nullptr;
    bm_status s = device_state(&st);
    if (s != BM_OK) return s;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return BM_ERR_CUDA;
    int code = 0;
    if (cudaMemcpy(&code, st->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return BM_ERR_CUDA;
    if (code != 0 && cudaMemset(st->status, 0, sizeof(int)) != cudaSuccess) return BM_ERR_CUDA;
    return static_cast<bm_status>(code);
}

void bm_set_wait_timeout_ms(uint32_t ms) { g_timeout_ms.store(ms == 0 ? 1 : ms); }

void bm_debug_inject_stall(int enable) { g_debug_stall.store(enable ? 1 : 0); }

bm_status bm_set_tile_override(int variant)
{
    if (variant < 0 || variant > 3) return BM_ERR_INVALID_VALUE;  // 0 = automatic, 1 + kSingle256 .. kPair256
    g_tile_override.store(variant);
    return BM_OK;
}

const char *bm_status_string(bm_status status)
{
    switch (status) {
    case BM_OK: return "BM_OK";
    case BM_ERR_INVALID_VALUE: return "BM_ERR_INVALID_VALUE";
    case BM_ERR_MISALIGNED: return "BM_ERR_MISALIGNED";
    case BM_ERR_ARCH: return "BM_ERR_ARCH";
    case BM_ERR_CUDA: return "BM_ERR_CUDA";
    case BM_ERR_TIMEOUT: return "BM_ERR_TIMEOUT";
    case BM_ERR_WORKSPACE: return "BM_ERR_WORKSPACE";
    }
    return "BM_ERR_UNKNOWN";
}

int bm_version(void) { return 100; }

}  // extern "C"
