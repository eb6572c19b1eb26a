// gemm_prefill.cu -- base product with the low-rank expand, for prefill-sized
// batches (compute bound: a 16384 x 14336 x 4096 GEMM is ~2 TFLOP). Two kernels:
// gemm_prefill_pair_kernel (clusters of two CTAs, 256-token tiles; above 128 tokens,
// described further down) and gemm_prefill_kernel (one CTA per 128-token tile):
//
// Persistent kernel, one CTA per SM, output tiles of 128 tokens x 256 columns
// walked in a grouped order (16 token tiles share one sweep over the columns,
// so their X rows stay in L2 while W streams).
//  * warp 8: TMA producer. Per 64-wide k-block it loads X[128 x 64] and
//    W[256 x 64] (128-byte swizzle) into a 4-stage ring (48 KB per stage).
//  * warp 9: MMA issuer. tcgen05.mma M=128 N=256 K=16, four per k-block, into
//    one of two TMEM accumulators (2 x 256 columns = all 512), so the
//    epilogue of tile i overlaps the MMAs of tile i+1.
//  * The expand Y += s_i (X A_i) B_i runs on the tensor cores too: when every
//    token of a tile with an adapter uses the same adapter (always, for
//    sequences of one adapter that start on a 128-token boundary), the
//    producer appends ceil(pages/4) k-blocks, each holding 32 rank columns: the
//    shrink's bf16 hi/lo pairs s*V = hi + lo of the tile's tokens (one TMA box
//    of 64 columns = [hi 32 | lo 32]; rows of base-only tokens are zero) and
//    four 4 KB slices of the adapter's interleaved B pages (bulk copies; a B
//    page is already a K-major no-swizzle operand: 8 columns x 16 bytes per
//    core matrix). Four MMAs per such block: hi and lo against the same B.
//    The product is accumulated in fp32 with the base product, so Y is rounded
//    once. Expand work: 2 * 32 / 64 = one k-block per 32 rank columns.
//  * warps 0-7: epilogue. Warp w reads TMEM lanes 32*(w%4).. (its 32 token
//    rows) and columns 128*(w/4).. in chunks of 32 with tcgen05.ld, rounds to
//    bf16 and stores Y. For a tile whose tokens use more than one adapter the
//    expand is added here instead, on CUDA cores (B pages read 16 bytes = 8
//    rank rows per column), before the rounding.
#include <mutex>

#include "device_common.cuh"

namespace lora {

namespace {

constexpr int kThreads = 320;
constexpr int kBM = 128, kBN = 256, kBK = 64;
constexpr int kXTileBytes = kBM * kBK * 2;   // 16 KB
constexpr int kWTileBytes = kBN * kBK * 2;   // 32 KB
constexpr int kStageBytes = kXTileBytes + kWTileBytes;
constexpr int kStages = 4;
constexpr int kGroupM = 16;
constexpr int kEpiWarps = 8;
constexpr uint32_t kTmemCols = 512;
constexpr int kPagesPerBlock = 4;            // 32 rank columns per expand k-block
constexpr int kPageSliceBytes = kBN * 16;    // 256 columns x 8 rank rows of bf16

struct PrefillArgs {
    int T, d_in, d_out;
    int KB, tiles_m, tiles_n, num_tiles;
    const int32_t *ids;
    const int32_t *tile_info;
    const uint16_t *Vhl;
    int ldh;
    uint16_t *Y;
    int *err;
    uint64_t *trace;  // measurement hook (first entry, last exit), or nullptr
};

__device__ __forceinline__ void tile_coords(int tile, const PrefillArgs &a, int &m, int &n)
{
    const int per_group = kGroupM * a.tiles_n;
    const int g = tile / per_group;
    const int first_m = g * kGroupM;
    const int gm = min(kGroupM, a.tiles_m - first_m);
    const int local = tile - g * per_group;
    m = first_m + local % gm;
    n = local / gm;
}

// Adapter use of one token tile (from the segment builder's tile table): mode 0 =
// no token has an adapter, 1 = one adapter (slot), 2 = several adapters (expand
// on CUDA cores).
struct TileLora {
    int mode, slot, npages, blocks;
    const int32_t *pages;
};

// Checked build: a tile's slot and page count within the pool (else no expand).
__device__ __forceinline__ bool tile_slot_ok(int slot, const PoolDev &pool, int *err)
{
#ifdef LORA_CHECK
    if (!check_range(slot, 0, pool.max_adapters, err)) return false;
    return check_range(pool.slots[(size_t)slot * pool.slot_stride + SLOT_NPAGES], 0, pool.max_pages + 1, err);
#else
    return true;
#endif
}

__device__ __forceinline__ TileLora tile_lora(int m, const PrefillArgs &a, const PoolDev &pool)
{
    TileLora r{0, -1, 0, 0, nullptr};
    if (a.tile_info == nullptr) return r;
    const int ti = a.tile_info[m];
    if (ti == kTileNoAdapter) return r;
    if (ti == kTileMixed) {
        r.mode = 2;
        return r;
    }
    if (!tile_slot_ok(ti, pool, a.err)) return r;
    const int32_t *row = pool.slots + (size_t)ti * pool.slot_stride;
    r.mode = 1;
    r.slot = ti;
    r.npages = row[SLOT_NPAGES];
    r.blocks = (r.npages + kPagesPerBlock - 1) / kPagesPerBlock;
    r.pages = row + SLOT_PAGES;
    return r;
}

// acc[j] += vv . (the 8 rank values of column ncol + j of a B page) for 32 columns;
// columns past d_out add nothing. The B words are loaded 16 at a time before any of
// them is used, so that a batch's loads are in flight together.
__device__ __forceinline__ void expand_page_32(float (&acc)[32], const float (&vv)[8], const uint16_t *bp,
                                               int ncol, int d_out)
{
#pragma unroll
    for (int j0 = 0; j0 < 32; j0 += 16) {
        uint4 b[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
            b[j] = ncol + j0 + j < d_out ? ldg_nc_v4(bp + (j0 + j) * kRankPage) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int j = 0; j < 16; ++j) acc[j0 + j] = dot8_f32_bf16(vv, b[j], acc[j0 + j]);
    }
}

// The B words of one row's expand for the warp's 128 columns starting at c0 (2 KB
// contiguous per page) into L2, one bulk prefetch per page, so that the gathers of the
// expand hit L2.
__device__ __forceinline__ void prefetch_row_b(const int32_t *pages, int np, int c0, const PrefillArgs &a,
                                               const PoolDev &pool)
{
    if (np <= 0 || c0 >= a.d_out) return;
    const uint32_t bytes = (uint32_t)min(128, a.d_out - c0) * 16u;
    for (int q = 0; q < np; ++q) {
        const int page = LORA_CHECKED(pages[q], 0, pool.num_pages, a.err, 0);
        prefetch_l2_bulk(pool.B_pages + ((size_t)page * a.d_out + c0) * kRankPage, bytes);
    }
}

// One epilogue warp's share of a finished accumulator: TMEM lanes 32*quarter.. (token
// rows t = row0 + lane), columns 128*half.. of the tile at column n0, in chunks of 32;
// with `own_expand`, each row's adapter expand added on CUDA cores; rounded to bf16
// and stored.
__device__ __forceinline__ void epilogue_rows(uint32_t tmem_buf, int quarter, int half, int row0, int n0,
                                              bool own_expand, const PrefillArgs &a, const PoolDev &pool)
{
    const int lane = threadIdx.x & 31;
    const int t = row0 + lane;
    const bool row_ok = t < a.T;
    int np = 0;
    const int32_t *pages = nullptr;
    const uint16_t *hrow = nullptr;
    if (own_expand && row_ok) {  // several adapters: this row's own expand
        const int id = a.ids[t];
        if (slot_loaded(pool.slots, pool.slot_stride, pool.max_adapters, id)) {
            const int32_t *row = pool.slots + (size_t)id * pool.slot_stride;
            np = row[SLOT_NPAGES];
            pages = row + SLOT_PAGES;
            hrow = a.Vhl + (size_t)t * a.ldh;
        }
    }
    prefetch_row_b(pages, np, n0 + half * 128, a, pool);
    uint16_t *yrow = a.Y + (size_t)t * a.d_out;
#pragma unroll 1
    for (int ch = 0; ch < 4; ++ch) {
        const int col0 = half * 128 + ch * 32;
        const int ncol = n0 + col0;
        uint32_t r[32];
        tmem_ld32_wait(tmem_buf + ((uint32_t)(quarter * 32) << 16) + (uint32_t)col0, r);
        float acc[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) acc[j] = __uint_as_float(r[j]);
        for (int q = 0; q < np; ++q) {
            const uint16_t *g = hrow + (q / 4) * 64 + (q % 4) * 8;
            const uint4 h = *reinterpret_cast<const uint4 *>(g);
            const uint4 l = *reinterpret_cast<const uint4 *>(g + 32);
            const float vv[8] = {bf16_lo(h.x) + bf16_lo(l.x), bf16_hi(h.x) + bf16_hi(l.x),
                                 bf16_lo(h.y) + bf16_lo(l.y), bf16_hi(h.y) + bf16_hi(l.y),
                                 bf16_lo(h.z) + bf16_lo(l.z), bf16_hi(h.z) + bf16_hi(l.z),
                                 bf16_lo(h.w) + bf16_lo(l.w), bf16_hi(h.w) + bf16_hi(l.w)};
            const uint16_t *bp = pool.B_pages + ((size_t)LORA_CHECKED(pages[q], 0, pool.num_pages, a.err, 0) * a.d_out + ncol) * kRankPage;
            expand_page_32(acc, vv, bp, ncol, a.d_out);
        }
        if (row_ok) {
#pragma unroll
            for (int j = 0; j < 32; j += 8) {
                if (ncol + j < a.d_out) {
                    uint4 o;
                    o.x = pack_bf16x2(acc[j + 0], acc[j + 1]);
                    o.y = pack_bf16x2(acc[j + 2], acc[j + 3]);
                    o.z = pack_bf16x2(acc[j + 4], acc[j + 5]);
                    o.w = pack_bf16x2(acc[j + 6], acc[j + 7]);
                    *reinterpret_cast<uint4 *>(yrow + ncol + j) = o;
                }
            }
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_prefill_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                        const __grid_constant__ CUtensorMap tmV, PrefillArgs a, PoolDev pool)
{
    trace_enter_released(a.trace);
    extern __shared__ uint8_t pre_smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(pre_smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)kStages * kStageBytes);
    uint64_t *empty = full + kStages;
    uint64_t *acc_full = empty + kStages;  // [2]
    uint64_t *acc_empty = acc_full + 2;    // [2]
    uint64_t *drain = acc_empty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_empty[i], kEpiWarps);
        }
        mbar_init(drain, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 9) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    if (warp == 8 && lane == 0) {
        tma_prefetch_map(&tmX);
        tma_prefetch_map(&tmW);
        tma_prefetch_map(&tmV);
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == 8) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int it = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < a.num_tiles && ok; tile += gridDim.x) {
                int m, n;
                tile_coords(tile, a, m, n);
                const TileLora tl = tile_lora(m, a, pool);
                const int steps = a.KB + (tl.mode == 1 ? tl.blocks : 0);
                const int n0 = n * kBN;
                const uint32_t slice_bytes = (uint32_t)min(kBN, a.d_out - n0) * 16u;
                for (int kb = 0; kb < steps; ++kb, ++it) {
                    const int s = it % kStages;
                    ok = mbar_wait(&empty[s], ((uint32_t)(it / kStages) & 1u) ^ 1u, &abort_flag, a.err);
                    if (!ok) break;
                    uint8_t *xs = smem + (size_t)s * kStageBytes;
                    if (kb < a.KB) {
                        mbar_arrive_expect_tx(&full[s], kStageBytes);
                        tma_load_2d(xs, &tmX, &full[s], kb * kBK, m * kBM);
                        tma_load_2d(xs + kXTileBytes, &tmW, &full[s], kb * kBK, n0);
                    } else {
                        const int e = kb - a.KB;
                        mbar_arrive_expect_tx(&full[s], kXTileBytes + kPagesPerBlock * slice_bytes);
                        tma_load_2d(xs, &tmV, &full[s], e * 64, m * kBM);
                        for (int i = 0; i < kPagesPerBlock; ++i) {
                            const int q = e * kPagesPerBlock + i;
                            const int page = q < tl.npages
                                                 ? LORA_CHECKED(tl.pages[q], 0, pool.num_pages, a.err, 0)
                                                 : 0;  // page 0 is zeros
                            bulk_load(xs + kXTileBytes + i * kPageSliceBytes,
                                      pool.B_pages + ((size_t)page * a.d_out + n0) * kRankPage,
                                      slice_bytes, &full[s]);
                        }
                    }
                }
            }
            for (int i = 0; i < kStages && i < it; ++i) {
                const int j = it - 1 - i;
                int dummy = 0;
                mbar_wait(&full[j % kStages], (uint32_t)(j / kStages) & 1u, &dummy, a.err);
            }
        }
        __syncwarp();
    } else if (warp == 9) {
        // ----------------------------------------------------------------- MMA
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(kBM, kBN);
            int it = 0, tc = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < a.num_tiles && ok; tile += gridDim.x, ++tc) {
                int m, n;
                tile_coords(tile, a, m, n);
                const TileLora tl = tile_lora(m, a, pool);
                const int steps = a.KB + (tl.mode == 1 ? tl.blocks : 0);
                const int buf = tc & 1;
                ok = mbar_wait(&acc_empty[buf], ((uint32_t)(tc >> 1) & 1u) ^ 1u, &abort_flag, a.err);
                if (!ok) break;
                tc_fence_after_sync();
                const uint32_t d = tmem + (uint32_t)(buf * kBN);
                for (int kb = 0; kb < steps; ++kb, ++it) {
                    const int s = it % kStages;
                    ok = mbar_wait(&full[s], (uint32_t)(it / kStages) & 1u, &abort_flag, a.err);
                    if (!ok) break;
                    tc_fence_after_sync();
                    const uint32_t xa = smem_u32(smem + (size_t)s * kStageBytes);
                    const uint32_t wa = xa + kXTileBytes;
                    if (kb < a.KB) {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_bf16_ss(d, sdesc_k_sw128(xa + kk * 32), sdesc_k_sw128(wa + kk * 32),
                                        idesc, (kb | kk) != 0);
                    } else {
                        // A: [hi j0..15 | hi j16..31 | lo j0..15 | lo j16..31]; B: page slices
                        // (0,1) hold j0..15, (2,3) hold j16..31. When the block's pages 2,3
                        // are past the adapter (zero pages), their two K-steps add nothing.
                        const bool upper = (kb - a.KB) * kPagesPerBlock + 2 < tl.npages;
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            if (!(kk & 1) || upper)
                                mma_bf16_ss(d, sdesc_k_sw128(xa + kk * 32),
                                            sdesc_k_none(wa + (kk & 1) * 2 * kPageSliceBytes,
                                                         kPageSliceBytes, 128),
                                            idesc, 1u);
                    }
                    mma_commit(&empty[s]);
                }
                if (ok) mma_commit(&acc_full[buf]);
            }
            mma_commit(drain);
            int dummy = 0;
            mbar_wait(drain, 0, &dummy, a.err);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int quarter = warp & 3, half = warp >> 2;
        int tc = 0;
        for (int tile = blockIdx.x; tile < a.num_tiles; tile += gridDim.x, ++tc) {
            int m, n;
            tile_coords(tile, a, m, n);
            const TileLora tl = tile_lora(m, a, pool);
            const int buf = tc & 1;
            bool ok = true;
            if (lane == 0) ok = mbar_wait(&acc_full[buf], (uint32_t)(tc >> 1) & 1u, &abort_flag, a.err);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after_sync();

            epilogue_rows(tmem + (uint32_t)(buf * kBN), quarter, half, m * kBM + quarter * 32, n * kBN,
                          tl.mode == 2, a, pool);
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[buf]);
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
    trace_exit(a.trace);
}

// ------------------------------------------------------------ CTA-pair variant
//
// A cluster of two CTAs computes a 256-token x 256-column tile with tcgen05 MMAs of
// cta_group::2 (M = 256, N = 256, K = 16): CTA r holds tokens r*128.. of the tile
// (its A half, and those rows of D in its TMEM) and W rows n0 + r*128.. (its half of
// B). Per k-block each CTA stages 16 KB of X and 16 KB of W (32 KB instead of 48 KB
// for 128 x 256 on one SM). A pipeline stage holds two k-blocks (three 64 KB stages):
// the tensor pipe was found waiting on the barrier round trip of each stage (wait,
// MMAs, commit), and eight MMAs per round trip instead of four raised its activity
// from 58 to 75 %. CTA 0 issues the MMAs; both CTAs' TMA loads complete on CTA 0's
// stage barrier; its commits are multicast to both CTAs' stage and accumulator
// barriers; both CTAs' epilogue warps release the accumulator on CTA 0's barrier.
// The epilogue stages each warp's 32 x 64 bf16 chunk in shared memory and writes it
// with a TMA store. The fused expand works as in the
// single-CTA kernel when every adapter token of the 256 uses one adapter: V rows of
// each half and each half's 128 columns of the adapter's B pages (one 2 KB TMA box
// per page: the B arena read as rows of 64 values, 16 rows a box).

// The pair kernel's epilogue for one warp: as epilogue_rows, but each 64-column chunk
// goes, as bf16, into a 128-byte-swizzled 32-row x 64-column staging tile in shared
// memory and leaves with one TMA store (rows past T and columns past d_out are not
// written), so Y reaches L2 in whole 128-byte row segments instead of 16-byte pieces
// of 32 rows at a time.
__device__ __forceinline__ void epilogue_rows_staged(uint32_t tmem_buf, int quarter, int half, int row0, int n0,
                                                     bool own_expand, const PrefillArgs &a, const PoolDev &pool,
                                                     uint8_t *ybuf, const CUtensorMap *tmY)
{
    const int lane = threadIdx.x & 31;
    const int t = row0 + lane;
    int np = 0;
    const int32_t *pages = nullptr;
    const uint16_t *hrow = nullptr;
    if (own_expand && t < a.T) {  // several adapters: this row's own expand
        const int id = a.ids[t];
        if (slot_loaded(pool.slots, pool.slot_stride, pool.max_adapters, id)) {
            const int32_t *row = pool.slots + (size_t)id * pool.slot_stride;
            np = row[SLOT_NPAGES];
            pages = row + SLOT_PAGES;
            hrow = a.Vhl + (size_t)t * a.ldh;
        }
    }
    prefetch_row_b(pages, np, n0 + half * 128, a, pool);
#pragma unroll 1
    for (int ch = 0; ch < 2; ++ch) {
        if (lane == 0) bulk_wait_read_all();  // the previous chunk's store has read ybuf
        __syncwarp();
#pragma unroll 1
        for (int sub = 0; sub < 2; ++sub) {
            const int col0 = half * 128 + ch * 64 + sub * 32;
            const int ncol = n0 + col0;
            uint32_t r[32];
            tmem_ld32_wait(tmem_buf + ((uint32_t)(quarter * 32) << 16) + (uint32_t)col0, r);
            float acc[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) acc[j] = __uint_as_float(r[j]);
            for (int q = 0; q < np; ++q) {
                const uint16_t *g = hrow + (q / 4) * 64 + (q % 4) * 8;
                const uint4 h = *reinterpret_cast<const uint4 *>(g);
                const uint4 l = *reinterpret_cast<const uint4 *>(g + 32);
                const float vv[8] = {bf16_lo(h.x) + bf16_lo(l.x), bf16_hi(h.x) + bf16_hi(l.x),
                                     bf16_lo(h.y) + bf16_lo(l.y), bf16_hi(h.y) + bf16_hi(l.y),
                                     bf16_lo(h.z) + bf16_lo(l.z), bf16_hi(h.z) + bf16_hi(l.z),
                                     bf16_lo(h.w) + bf16_lo(l.w), bf16_hi(h.w) + bf16_hi(l.w)};
                const uint16_t *bp = pool.B_pages + ((size_t)LORA_CHECKED(pages[q], 0, pool.num_pages, a.err, 0) * a.d_out + ncol) * kRankPage;
                expand_page_32(acc, vv, bp, ncol, a.d_out);
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                uint4 o;
                o.x = pack_bf16x2(acc[8 * k + 0], acc[8 * k + 1]);
                o.y = pack_bf16x2(acc[8 * k + 2], acc[8 * k + 3]);
                o.z = pack_bf16x2(acc[8 * k + 4], acc[8 * k + 5]);
                o.w = pack_bf16x2(acc[8 * k + 6], acc[8 * k + 7]);
                const int c = sub * 4 + k;  // 16-byte chunk of the 128-byte row
                *reinterpret_cast<uint4 *>(ybuf + lane * 128 + ((c ^ (lane & 7)) << 4)) = o;
            }
        }
        fence_proxy_async_smem();
        __syncwarp();
        const int x = n0 + half * 128 + ch * 64;
        if (lane == 0 && x < a.d_out && row0 < a.T) tma_store_2d(tmY, ybuf, x, row0);
    }
}

constexpr int kPBM = 256;                     // tokens per pair tile (128 per CTA)
constexpr int kPHalfBytes = 128 * kBK * 2;    // 16 KB: one CTA's X or W half of a k-block
constexpr int kPBlockBytes = 2 * kPHalfBytes;  // one k-block of one CTA: X half + W half
constexpr int kPKps = 2;                       // k-blocks per pipeline stage
constexpr int kPStageBytes = kPKps * kPBlockBytes;
constexpr int kPStages = 3;
constexpr int kPGroupM = 16;                  // 16 x 256 tokens share one column sweep
constexpr int kPSliceBytes = 128 * 16;        // 128 columns x 8 rank values of one page
constexpr int kPYStageBytes = 32 * 128;       // one epilogue warp's 32 x 64 bf16 staging tile
constexpr size_t kPairSmem =
    1024 + (size_t)kPStages * kPStageBytes + kEpiWarps * kPYStageBytes + (2 * kPStages + 5) * 8 + 16;

__device__ __forceinline__ void pair_tile_coords(int tile, const PrefillArgs &a, int &m, int &n)
{
    const int tiles_m = (a.T + kPBM - 1) / kPBM;
    const int per_group = kPGroupM * a.tiles_n;
    const int g = tile / per_group;
    const int first_m = g * kPGroupM;
    const int gm = min(kPGroupM, tiles_m - first_m);
    const int local = tile - g * per_group;
    m = first_m + local % gm;
    n = local / gm;
}

// Adapter use of a pair tile: the tensor-core expand (mode 1) when every token of the
// 256 that has an adapter uses the same one; otherwise each CTA adds its own rows'
// expand in the epilogue (own_expand) where its 128-token half has adapters.
__device__ __forceinline__ TileLora pair_tile_lora(int m, uint32_t rank, const PrefillArgs &a,
                                                   const PoolDev &pool, bool &own_expand)
{
    own_expand = false;
    TileLora r{0, -1, 0, 0, nullptr};
    if (a.tile_info == nullptr) return r;
    const int i0 = a.tile_info[2 * m];
    const int i1 = 2 * m + 1 < a.tiles_m ? a.tile_info[2 * m + 1] : kTileNoAdapter;
    int slot = -1;
    bool single = true;
    for (int k = 0; k < 2; ++k) {
        const int ti = k ? i1 : i0;
        if (ti == kTileMixed) single = false;
        else if (ti >= 0) {
            if (slot < 0) slot = ti;
            else if (slot != ti) single = false;
        }
    }
    if (!single) {
        own_expand = (rank ? i1 : i0) != kTileNoAdapter;
        return r;
    }
    if (slot < 0) return r;
    if (!tile_slot_ok(slot, pool, a.err)) return r;
    const int32_t *row = pool.slots + (size_t)slot * pool.slot_stride;
    r.mode = 1;
    r.slot = slot;
    r.npages = row[SLOT_NPAGES];
    r.blocks = (r.npages + kPagesPerBlock - 1) / kPagesPerBlock;
    r.pages = row + SLOT_PAGES;
    return r;
}

// A pair tile's coordinates and adapter use; each role loads the next tile's while the
// current one runs, so the dependent table loads stay off the tile boundary.
struct PairTile {
    int m, n;
    TileLora tl;
    bool own;
};

__device__ __forceinline__ PairTile pair_tile(int tile, int tiles, uint32_t rank, const PrefillArgs &a,
                                              const PoolDev &pool)
{
    PairTile r{0, 0, TileLora{0, -1, 0, 0, nullptr}, false};
    if (tile >= tiles) return r;
    pair_tile_coords(tile, a, r.m, r.n);
    r.tl = pair_tile_lora(r.m, rank, a, pool, r.own);
    return r;
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_prefill_pair_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                             const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmB,
                             const __grid_constant__ CUtensorMap tmY, PrefillArgs a, PoolDev pool)
{
    trace_enter_released(a.trace);
    extern __shared__ uint8_t pre_smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(pre_smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *ystage = smem + (size_t)kPStages * kPStageBytes;  // [kEpiWarps][32 x 128 B]
    uint64_t *full = reinterpret_cast<uint64_t *>(ystage + kEpiWarps * kPYStageBytes);
    uint64_t *empty = full + kPStages;
    uint64_t *acc_full = empty + kPStages;  // [2]
    uint64_t *acc_empty = acc_full + 2;     // [2], used in CTA 0
    uint64_t *drain = acc_empty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_cta_rank();
    const int cluster = (int)blockIdx.x >> 1, clusters = (int)gridDim.x >> 1;
    const int tiles = ((a.T + kPBM - 1) / kPBM) * a.tiles_n;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kPStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_empty[i], 2 * kEpiWarps);
        }
        mbar_init(drain, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 9) {
        tmem_alloc_pair(tmem_slot, kTmemCols);
        tmem_relinquish_pair();
    }
    if (warp == 8 && lane == 0) {
        tma_prefetch_map(&tmX);
        tma_prefetch_map(&tmW);
        tma_prefetch_map(&tmV);
        tma_prefetch_map(&tmB);
        tma_prefetch_map(&tmY);
    }
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync_all();  // both CTAs' barriers exist before either signals the other's
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == 8) {
        // ------------------------------------------- producer (both CTAs, own halves)
        if (lane == 0) {
            int it = 0;
            bool ok = true;
            PairTile cur = pair_tile(cluster, tiles, rank, a, pool);
            for (int tile = cluster; tile < tiles && ok; tile += clusters) {
                const PairTile nxt = pair_tile(tile + clusters, tiles, rank, a, pool);
                const TileLora &tl = cur.tl;
                const int ne = tl.mode == 1 ? tl.blocks : 0;
                const int sb = (a.KB + kPKps - 1) / kPKps, steps = sb + (ne + kPKps - 1) / kPKps;
                const int n0 = cur.n * kBN + (int)rank * 128;   // this CTA's W rows / B columns
                const int r0 = cur.m * kPBM + (int)rank * 128;  // this CTA's token rows
                // the first expand block's page numbers, loaded now and used after the
                // base k-blocks (each copy is an asm statement that keeps its place, so
                // a load written beside it would hold up the producer for its latency)
                int pg0[kPagesPerBlock];
#pragma unroll
                for (int i = 0; i < kPagesPerBlock; ++i) pg0[i] = ne > 0 && i < tl.npages ? tl.pages[i] : 0;
                for (int st = 0; st < steps; ++st, ++it) {
                    const int s = it % kPStages;
                    ok = mbar_wait_cluster(&empty[s], ((uint32_t)(it / kPStages) & 1u) ^ 1u, &abort_flag,
                                           a.err);
                    if (!ok) break;
                    const uint32_t fb = cluster_map(&full[s], 0);
                    uint8_t *xs = smem + (size_t)s * kPStageBytes;
                    if (st < sb) {
                        const int k0 = st * kPKps, nk = min(kPKps, a.KB - k0);
                        if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * nk * kPBlockBytes);
                        for (int j = 0; j < nk; ++j) {
                            tma_load_2d_pair(xs + j * kPBlockBytes, &tmX, fb, (k0 + j) * kBK, r0);
                            tma_load_2d_pair(xs + j * kPBlockBytes + kPHalfBytes, &tmW, fb, (k0 + j) * kBK, n0);
                        }
                    } else {
                        const int e0 = (st - sb) * kPKps, nj = min(kPKps, ne - e0);
                        if (rank == 0)
                            mbar_arrive_expect_tx(&full[s], 2 * nj * (kPHalfBytes + kPagesPerBlock * kPSliceBytes));
                        for (int j = 0; j < nj; ++j) {
                            const int e = e0 + j;
                            uint8_t *bs = xs + j * kPBlockBytes;
                            // the block's page numbers (page 0 is zeros), all loaded before
                            // the first copy is issued
                            int pg[kPagesPerBlock];
#pragma unroll
                            for (int i = 0; i < kPagesPerBlock; ++i) {
                                const int q = e * kPagesPerBlock + i;
                                pg[i] = e == 0 ? pg0[i] : q < tl.npages ? tl.pages[q] : 0;
                            }
                            tma_load_2d_pair(bs, &tmV, fb, e * 64, r0);
#pragma unroll
                            for (int i = 0; i < kPagesPerBlock; ++i) {
                                const int page = LORA_CHECKED(pg[i], 0, pool.num_pages, a.err, 0);
                                // columns n0.. of the page: 128 x 16 B from row (page d_out + n0) / 8
                                // of the 128-byte-row view (n0 and d_out are multiples of 8)
                                tma_load_2d_pair(bs + kPHalfBytes + i * kPSliceBytes, &tmB, fb, 0,
                                                 (int)(((long long)page * a.d_out + n0) >> 3));
                            }
                        }
                    }
                }
                cur = nxt;
            }
            // CTA 0's stage barriers count both CTAs' copies: do not leave while any is
            // in flight
            for (int i = 0; rank == 0 && i < kPStages && i < it; ++i) {
                const int j = it - 1 - i;
                int dummy = 0;
                mbar_wait_cluster(&full[j % kPStages], (uint32_t)(j / kPStages) & 1u, &dummy, a.err);
            }
        }
        __syncwarp();
    } else if (warp == 9) {
        // ------------------------------------------------------- MMA (CTA 0 only)
        if (lane == 0 && rank == 0) {
            const uint32_t idesc = idesc_bf16_f32(kPBM, kBN);
            int it = 0, tc = 0;
            bool ok = true;
            PairTile cur = pair_tile(cluster, tiles, rank, a, pool);
            for (int tile = cluster; tile < tiles && ok; tile += clusters, ++tc) {
                const PairTile nxt = pair_tile(tile + clusters, tiles, rank, a, pool);
                const int ne = cur.tl.mode == 1 ? cur.tl.blocks : 0;
                const int sb = (a.KB + kPKps - 1) / kPKps, steps = sb + (ne + kPKps - 1) / kPKps;
                const int buf = tc & 1;
                ok = mbar_wait_cluster(&acc_empty[buf], ((uint32_t)(tc >> 1) & 1u) ^ 1u, &abort_flag, a.err);
                if (!ok) break;
                tc_fence_after_sync();
                const uint32_t d = tmem + (uint32_t)(buf * kBN);
                for (int st = 0; st < steps; ++st, ++it) {
                    const int s = it % kPStages;
                    ok = mbar_wait_cluster(&full[s], (uint32_t)(it / kPStages) & 1u, &abort_flag, a.err);
                    if (!ok) break;
                    tc_fence_after_sync();
                    const uint32_t sa = smem_u32(smem + (size_t)s * kPStageBytes);
                    if (st < sb) {
                        const int nk = min(kPKps, a.KB - st * kPKps);
#pragma unroll
                        for (int j = 0; j < kPKps; ++j) {
                            if (j >= nk) break;
                            const uint32_t xa = sa + j * kPBlockBytes, wa = xa + kPHalfBytes;
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                mma_bf16_ss_pair(d, sdesc_k_sw128(xa + kk * 32), sdesc_k_sw128(wa + kk * 32),
                                                 idesc, (st | j | kk) != 0);
                        }
                    } else {
                        const int nj = min(kPKps, ne - (st - sb) * kPKps);
#pragma unroll
                        for (int j = 0; j < kPKps; ++j) {
                            if (j >= nj) break;
                            const uint32_t xa = sa + j * kPBlockBytes, wa = xa + kPHalfBytes;
                            // (the single-CTA kernel's layout; the zero pages' K-steps skipped)
                            const int e = (st - sb) * kPKps + j;
                            const bool upper = e * kPagesPerBlock + 2 < cur.tl.npages;
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                if (!(kk & 1) || upper)
                                    mma_bf16_ss_pair(d, sdesc_k_sw128(xa + kk * 32),
                                                     sdesc_k_none(wa + (kk & 1) * 2 * kPSliceBytes, kPSliceBytes, 128),
                                                     idesc, 1u);
                        }
                    }
                    mma_commit_pair(&empty[s], 0x3);
                }
                if (ok) mma_commit_pair(&acc_full[buf], 0x3);
                cur = nxt;
            }
            mma_commit_pair(drain, 0x1);
            int dummy = 0;
            mbar_wait(drain, 0, &dummy, a.err);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------- epilogue (both CTAs, own rows)
        const int quarter = warp & 3, half = warp >> 2;
        const uint32_t release = 0;  // CTA 0 holds the accumulator barriers' empty side
        int tc = 0;
        PairTile cur = pair_tile(cluster, tiles, rank, a, pool);
        for (int tile = cluster; tile < tiles; tile += clusters, ++tc) {
            const PairTile t = cur;
            cur = pair_tile(tile + clusters, tiles, rank, a, pool);
            const int m = t.m, n = t.n;
            const bool own = t.own;
            const int buf = tc & 1;
            bool ok = true;
            if (lane == 0)
                ok = mbar_wait_cluster(&acc_full[buf], (uint32_t)(tc >> 1) & 1u, &abort_flag, a.err);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after_sync();
            epilogue_rows_staged(tmem + (uint32_t)(buf * kBN), quarter, half,
                                 m * kPBM + (int)rank * 128 + quarter * 32, n * kBN, own, a, pool,
                                 ystage + warp * kPYStageBytes, &tmY);
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(cluster_map(&acc_empty[buf], release));
        }
        if (lane == 0) bulk_wait_all();  // this warp's stores of Y have completed
        __syncwarp();
    }

    tc_fence_before_sync();
    __syncthreads();
    cluster_sync_all();  // neither CTA leaves while the other may still use its memory
    if (warp == 9) {
        tc_fence_after_sync();
        tmem_dealloc_pair(tmem, kTmemCols);
    }
    trace_exit(a.trace);
}

// Clusters of the pair kernel that can be resident at once on the current device
// (clusters sit within one GPC, so this can be below half the SMs).
int pair_clusters(size_t smem, int num_sms)
{
    static int cached[64];
    static std::once_flag once[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return num_sms / 2;
    std::call_once(once[dev], [&] {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * (num_sms / 2));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, (const void *)gemm_prefill_pair_kernel, &cfg) != cudaSuccess ||
            n < 1) {
            cudaGetLastError();
            n = num_sms / 2;
        }
        cached[dev] = n < num_sms / 2 ? n : num_sms / 2;
    });
    return cached[dev] > 0 ? cached[dev] : 1;
}

cudaError_t launch_pair(const CUtensorMap &tmX, const CUtensorMap &tmW, const CUtensorMap &tmV,
                        const CUtensorMap &tmB, const CUtensorMap &tmY, const PrefillArgs &a, const PoolDev &pool,
                        int num_sms, cudaStream_t stream)
{
    const size_t smem = kPairSmem;
    cudaError_t e = ensure_smem_attr((const void *)gemm_prefill_pair_kernel, smem);
    if (e != cudaSuccess) return e;
    const int tiles = ((a.T + kPBM - 1) / kPBM) * a.tiles_n;
    int clusters = pair_clusters(smem, num_sms);
    if (clusters > tiles) clusters = tiles;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * clusters);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemm_prefill_pair_kernel, tmX, tmW, tmV, tmB, tmY, a, pool);
}

}  // namespace

cudaError_t launch_gemm_prefill(const CUtensorMap &tmX, const CUtensorMap &tmW,
                                const CUtensorMap &tmV, const CUtensorMap *tmB, const CUtensorMap *tmY, int T,
                                const int32_t *ids,
                                const int32_t *tile_info, const PoolDev &pool, const uint16_t *Vhl, int ldh, uint16_t *Y,
                                int num_sms, int *err, cudaStream_t stream, uint64_t *trace)
{
    PrefillArgs a{};
    a.trace = trace;
    a.T = T;
    a.d_in = pool.d_in;
    a.d_out = pool.d_out;
    a.KB = (pool.d_in + kBK - 1) / kBK;
    a.tiles_m = (T + kBM - 1) / kBM;
    a.tiles_n = (pool.d_out + kBN - 1) / kBN;
    a.num_tiles = a.tiles_m * a.tiles_n;
    a.ids = ids;
    a.tile_info = tile_info;
    a.Vhl = Vhl;
    a.ldh = ldh;
    a.Y = Y;
    a.err = err;
    if (a.num_tiles == 0) return cudaSuccess;
    if (tmB != nullptr) {
        if (tmY == nullptr) return cudaErrorInvalidValue;
        return launch_pair(tmX, tmW, tmV, *tmB, *tmY, a, pool, num_sms, stream);
    }
    const size_t smem = 1024 + (size_t)kStages * kStageBytes + (2 * kStages + 5) * 8 + 16;
    cudaError_t e = ensure_smem_attr((const void *)gemm_prefill_kernel, smem);
    if (e != cudaSuccess) return e;
    const int grid = a.num_tiles < num_sms ? a.num_tiles : num_sms;
    gemm_prefill_kernel<<<grid, kThreads, smem, stream>>>(tmX, tmW, tmV, a, pool);
    return cudaGetLastError();
}

}  // namespace lora
