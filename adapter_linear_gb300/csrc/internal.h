// internal.h -- constants, device-table layouts and kernel launchers shared by
// the translation units of the library (not part of the public ABI).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace lora {

// ---------------------------------------------------------------- pool layout
// Page = 8 rank rows of one adapter.
//   A arena: bf16 [num_pages][8][d_in]   (page q of adapter i holds columns
//            8q..8q+7 of A_i, transposed: row jj = A_i[:, 8q+jj]).
//   B arena: bf16 [num_pages][d_out][8]  (page q holds rows 8q..8q+7 of B_i,
//            interleaved: element [n][jj] = B_i[8q+jj, n]).
// Rank rows beyond an adapter's rank inside its last page are zero. Page 0 is
// an all-zero page that pads MMA operands to a multiple of 16 rank rows.
constexpr int kRankPage = 8;

// Slot table: int32 [max_adapters][slot_stride]
constexpr int SLOT_RANK = 0;     // rank (0 = empty slot); a chain: the members' ranks summed
constexpr int SLOT_NPAGES = 1;   // pages: ceil(rank / 8); a chain: the members' pages
constexpr int SLOT_SCALE = 2;    // alpha / rank as fp32 bits (a chain: its first member's)
constexpr int SLOT_MEMBERS = 3;  // a chain's member adapters (0: an adapter's own pages)
constexpr int SLOT_PAGES = 4;    // page ids, npages entries (up to max_pages), then one
                                 // fp32 scale per page at slot_page_scale(max_pages, q)
__host__ __device__ constexpr int slot_page_scale(int max_pages, int q)
{
    return SLOT_PAGES + max_pages + q;
}

// Segment-table header (int32 [4])
constexpr int HDR_NBASE = 0;    // tokens with id -1 (and invalid ids)
constexpr int HDR_NUMSEG = 1;   // segments (distinct loaded ids present)
constexpr int HDR_UNITS = 2;    // sum over segments of ceil(len / kShrinkRows)

constexpr int kShrinkRows = 128;       // token rows per tensor-core shrink unit
constexpr int kShrinkSmallSeg = 16;    // segments of at most this many tokens: warp-level shrink
constexpr int kDecodeMaxT = 256;       // largest batch of the decode path
constexpr int kAutoDecodeMaxT = 512;   // AUTO runs larger batches up to this in decode slices

// Device error word bits.
constexpr int kErrBadIdBit = 1;
constexpr int kErrTimeoutBit = 2;
constexpr int kErrRangeBit = 4;   // checked build (LORA_CHECK): an index out of range

// Every mbarrier wait gives up after this long (then flags kErrTimeoutBit).
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;

struct SegTables {
    int32_t *order;      // [T]
    int32_t *hdr;        // [4]
    int32_t *seg_start;  // [max_seg + 1]
    int32_t *seg_slot;   // [max_seg]
    int32_t *seg_ublk;   // [max_seg + 1]  prefix of ceil(len / kShrinkRows)
    int32_t *tile_info;  // [ceil(T / 128)]  adapters of each 128-token tile in token
                         // order: the slot if all its tokens with an adapter share one,
                         // kTileNoAdapter, or kTileMixed
    // the multi-CTA builder's scratch (nullptr: the single-CTA builder runs)
    int32_t *keys;       // [T] sort key of every token (id + 1, 0 = base only)
    int32_t *chist;      // [chunks][K] tokens per (chunk, key), then [K] first position per key
    int32_t *ticket;     // [1] chunks done (zero between calls)
};
constexpr int kSegChunk = 256;       // tokens per CTA of the multi-CTA segment builder
constexpr int kSegMultiMaxKeys = 4097;  // keys (max_adapters + 1) it can take (scratch sized for them)
// it runs for pools of up to kSegMultiKeys keys, or batches of kSegMultiMinT tokens and
// more; else the single-CTA builder (measured with 2001 keys: 256 tokens 7 vs 16 us,
// 4096 tokens 26 vs 23 us)
constexpr int kSegMultiKeys = 1024;
constexpr int kSegMultiMinT = 2048;
constexpr int kTileNoAdapter = -1;
constexpr int kTileMixed = -2;

struct PoolDev {
    const uint16_t *A_pages;  // bf16 bits
    const uint16_t *B_pages;
    const int32_t *slots;
    int slot_stride;
    int max_adapters;
    int max_pages;            // pages per adapter at max_rank
    int num_pages;            // pages in each arena
    int d_in, d_out;
};

// ------------------------------------------------------------------ launchers

size_t seg_build_smem_bytes(int max_adapters, int warps);
// vhl != nullptr: also zero the rows [ldh] of vhl of tokens without an adapter.
// trace (here and below): the launch's four words of the measurement hook (see
// trace_enter in device_common.cuh), or nullptr.
cudaError_t launch_seg_build(const int32_t *ids, int T, const PoolDev &pool, SegTables tabs,
                             int *err, uint16_t *vhl, int ldh, cudaStream_t stream,
                             uint64_t *trace = nullptr);

// Prefill shrink (tcgen05), 128-token units per segment: writes s_i X[t,:] A_i as
// bf16 hi/lo pairs grouped per 32 rank columns (see shrink.cu) into Vhl [T][ldh].
// tmA: the A arena with a box of one page (8 rows x 64); tmAw: a box of
// round16(8 * max_pages) rows x 64 (consecutive pages in one copy).
cudaError_t launch_shrink_small(const uint16_t *X, int T, const PoolDev &pool, SegTables tabs, uint16_t *Vhl,
                                int ldh, int num_sms, int *err, cudaStream_t stream);
cudaError_t launch_shrink_tc(const CUtensorMap &tmX, const CUtensorMap &tmA,
                             const CUtensorMap &tmAw, const uint16_t *X,
                             int T, const PoolDev &pool, SegTables tabs, uint16_t *Vhl, int ldh,
                             int num_sms, int *err, cudaStream_t stream, uint64_t *trace = nullptr);

// ---------------------------------------------------------------- decode path
// One decode call covers 1..kMaxGroup problems that share the token ids (one
// lora_linear call, or the layers of one grouped call); their (tile, k-block)
// units are concatenated in problem order for the stream-K split.
constexpr int kMaxGroup = 8;

struct DecodeProblem {
    PoolDev pool;           // pool.slots == nullptr: no adapters (base product only)
    const uint16_t *X;      // [T][d_in]
    float *V;               // shrink output [T][ldv]
    int ldv;
    uint16_t *Y;            // [T][d_out]
    int *err;               // the pool's error word (bad ids)
    int KB;                 // 128-column k-blocks
    int n_tiles;            // 128-row tiles of d_out
    int u_begin;            // first unit of this problem
    int g_begin;            // first tile in the concatenated tile order
    int pair_begin;         // first shrink (token, page) pair
    int col_blk_begin;      // first block of the finishing grid
};

// The plan of one decode call: the fields below, then its problem table. Kernels
// take a copy sized for the problems it holds (NP = 1 for a single layer,
// kMaxGroup otherwise) to keep their parameter block small.
struct DecodePlanHead {
    int n, T, ntok;
    int U, G;               // units, CTAs (stream-K ranges)
    int grid;               // CTAs launched (>= G: the rest only run shrink pairs)
    int max_seg;            // most tiles one range touches (partials per CTA)
    int n_acc;              // TMEM accumulators in the ring
    int stages;
    int pairs;              // shrink pairs of all problems
    int col_blocks;         // finishing grid.x
    bool fin_two_pages;     // the finishing pass holds two B pages (else one) in registers
    bool tight;             // register-bounded kernel variants (see gemm_decode.cu)
    bool prefetch_a;        // A pages of the shrink pairs into L2 before the wait
    uint64_t *trace;        // measurement hook: LORA_KERNEL_SLOTS x 4 words (see trace_enter), or nullptr
    uint32_t tmem_cols;
    size_t smem_bytes;
    int raw_stages;         // 4-bit base: stages of the ring of codes (0: a bf16 base)
};

template <int NP>
struct DecodePlanT : DecodePlanHead {
    static constexpr int kNP = NP;
    DecodeProblem prob[NP];
};
using DecodePlan = DecodePlanT<kMaxGroup>;

template <int NP>
struct DecodeMapsT {
    CUtensorMap W[NP];  // W_m [d_out][d_in], box 64 x 128
    CUtensorMap X[NP];  // X_m [T][d_in], box 64 x ntok
};
using DecodeMaps = DecodeMapsT<kMaxGroup>;

// The 4-bit base (one layer): codes [d_out][d_in/2] bytes, box 64 B x 128 rows; scales
// [d_in/128][d_out] bf16 and zeros [d_in/128][d_out] bytes, boxes 128 x 1.
constexpr int kQ4Group = 128;
struct DecodeMapsQ4 {
    CUtensorMap Wq, S, Z, X;
};

// Shapes and the stream-K split (pointers left for the caller to fill);
// max_G bounds the number of ranges. False when the shapes are out of range.
bool plan_decode(int n, int T, const int *d_in, const int *d_out, const int *max_pages, int max_G,
                 DecodePlan *out);
size_t decode_partials_floats(const DecodePlan &p);
// Base products (stream-K partials) + the per-token shrink of every problem with a
// pool (ids == nullptr: no shrink). err takes the timeout bit.
cudaError_t launch_gemm_decode(const DecodeMaps &maps, const DecodePlan &plan, const int32_t *ids,
                               float *partials, int *err, cudaStream_t stream);
// The same kernel's plan and launch for a 4-bit base (one layer): the W tiles are
// dequantised in shared memory (plan_decode_q4 sets the stage counts; false when they
// do not fit).
bool plan_decode_q4(DecodePlan *plan);
cudaError_t launch_gemm_decode_q4(const DecodeMapsQ4 &maps, const DecodePlan &plan, const int32_t *ids,
                                  float *partials, int *err, cudaStream_t stream);
// The 4-bit base to bf16 [d_out][d_in] (prefill path; d_in % 128 == 0).
cudaError_t launch_dequant_q4(const uint8_t *Wq, const uint16_t *scales, const uint8_t *zeros, int d_out,
                              int d_in, uint16_t *W, cudaStream_t stream);
// Y_m = bf16(sum of split-K partials + s_i V_m[t] B_i); ids == nullptr: no branch.
// Launched with programmatic stream serialization after launch_gemm_decode.
cudaError_t launch_finish_decode(const DecodePlan &plan, const float *partials, const int32_t *ids,
                                 cudaStream_t stream);

// Prefill GEMM with the expand: tmV is a TMA map of Vhl [T x ldh] (box 128 x 64);
// tile_info from the segment builder; ids == nullptr: base product only.
// tmB == nullptr: one CTA per 128 x 256 tile (tmW box 256 x 64); else CTA pairs per
// 256 x 256 tile (tmW box 128 x 64, tmB the B arena's 128 x 8 boxes, tmY a map of Y
// with box 32 x 64).
cudaError_t launch_gemm_prefill(const CUtensorMap &tmX, const CUtensorMap &tmW,
                                const CUtensorMap &tmV, const CUtensorMap *tmB, const CUtensorMap *tmY, int T,
                                const int32_t *ids,
                                const int32_t *tile_info, const PoolDev &pool, const uint16_t *Vhl, int ldh, uint16_t *Y,
                                int num_sms, int *err, cudaStream_t stream, uint64_t *trace = nullptr);

// Pack a row-major A (d_in x rank) and B (rank x d_out) into pool pages.
cudaError_t launch_pack_adapter(const uint16_t *A, const uint16_t *B, int rank, const int32_t *pages,
                                int npages, const PoolDev &pool, uint16_t *A_pages,
                                uint16_t *B_pages, int *err, cudaStream_t stream);

// Host: on the current device, give a kernel the largest shared-memory carveout
// and raise its dynamic shared-memory limit to at least `bytes` (remembered
// per kernel and device, so repeated launches do not repeat the driver calls).
cudaError_t ensure_smem_attr(const void *kernel, size_t bytes);

// Host: build a 2-D bf16 TMA descriptor over a row-major [rows x inner] tensor, box
// [box_rows x box_inner], with 128-byte swizzle (or none: rows land box_inner * 2
// bytes apart).
bool make_tmap_bf16_2d(CUtensorMap *map, const void *base, uint64_t inner, uint64_t rows,
                       uint64_t row_pitch_bytes, uint32_t box_inner, uint32_t box_rows,
                       bool swizzle128 = true);
// The same for a byte tensor (no swizzle).
bool make_tmap_u8_2d(CUtensorMap *map, const void *base, uint64_t inner, uint64_t rows,
                     uint64_t row_pitch_bytes, uint32_t box_inner, uint32_t box_rows);

}  // namespace lora
