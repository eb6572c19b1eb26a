// shrink.cu -- the prefill path's low-rank "shrink" V = s_i * X[t,:] A_i for
// every token with an adapter: the low-dimensional intermediate that the
// LoRA-Land blog (核心实现解析 / 2) forms first, so that the extra work stays a
// small fraction of the base product. (The decode path computes it inside its
// GEMM kernel.) The scale s_i = alpha_i / r_i is folded in here.
//
// shrink_tc_kernel: persistent; one unit = up to 128 tokens of one segment
// (tokens grouped by adapter). tcgen05 MMA M=128 (tokens) x N=16..256 (rank
// rows, padded with the zero page) x K=d_in, operands staged by TMA (X rows
// when the segment's tokens are contiguous, else gathered by the producer warp
// into the same 128-byte-swizzled layout), fp32 accumulator in TMEM,
// double-buffered so one unit's epilogue overlaps the next unit's MMAs.
//
// Segments of at most kShrinkSmallSeg tokens, and segments whose tokens are not
// consecutive rows of X (a batch whose tokens are spread over many adapters), are left
// to shrink_small_kernel (warp-level MMAs on 16-token chunks): a 128-row tile holding a
// few tokens would still run the whole K loop here, and scattered rows would have to be
// gathered by one warp.
//
// Output Vhl, bf16 [T][ldh], row = token: each fp32 value v is stored as the
// pair hi = bf16(v), lo = bf16(v - hi) (hi + lo carries about 16 significant
// bits), grouped per 32 rank columns as [hi 0..31 | lo 0..31] [hi 32..63 | ...],
// so a 64-column TMA box is exactly the A operand of four MMA K-steps of the
// expand in the prefill GEMM. Columns past an adapter's rank, up to its last
// 32-column group, are written as zeros.
#include <algorithm>

#include "device_common.cuh"

namespace lora {

// ========================================================== tensor-core shrink

namespace {

constexpr int kTcThreads = 192;          // warps 0-3 epilogue, 4 producer, 5 MMA
constexpr int kXTileBytes = 128 * 128;   // 128 rows x 64 bf16
// Two 64-column boxes per pipeline stage (k-block = 128 columns): fewer barrier
// round trips per byte and twice the bytes in flight per stage.
constexpr int kSBoxes = 2;

struct UnitInfo {
    int p0, p1;       // positions in `order`
    int npages;       // adapter pages
    int n;            // MMA N: npages * 8 rounded up to 16
    const int32_t *pages;
    const int32_t *scales;  // fp32 bits, one per page (up to n / 8 entries readable)
};

// The segment of shrink unit u: the largest s with seg_ublk[s] <= u (seg_ublk ascending,
// [num_seg + 1]).
__device__ __forceinline__ int unit_segment(int u, const SegTables &tabs)
{
    int lo = 0, hi = tabs.hdr[HDR_NUMSEG];
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (tabs.seg_ublk[mid] <= u) lo = mid; else hi = mid;
    }
    return lo;
}

// Whether segment s runs on the warp-level shrink: at most kShrinkSmallSeg tokens, or
// tokens that are not consecutive rows (the order inside a segment ascends, so the
// rows are consecutive exactly when the last minus the first is the length minus one).
__device__ __forceinline__ bool seg_on_warp_shrink(int s, const SegTables &tabs)
{
    const int p0 = tabs.seg_start[s], len = tabs.seg_start[s + 1] - p0;
    return len <= kShrinkSmallSeg || tabs.order[p0 + len - 1] - tabs.order[p0] != len - 1;
}

// The tensor-core shrink's copy of the segments' unit prefix in shared memory, each entry
// with bit 31 set when the segment is left to the warp-level shrink ([nseg + 1], the last
// entry the number of units); nullptr when it did not fit (the global tables are read).
constexpr uint32_t kSmallBit = 0x80000000u;

__device__ __forceinline__ int unit_segment_smem(int u, const uint32_t *sseg, int nseg)
{
    int lo = 0, hi = nseg;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if ((int)(sseg[mid] & ~kSmallBit) <= u) lo = mid; else hi = mid;
    }
    return lo;
}

// Whether unit u belongs to a segment the warp-level shrink takes (every role of the
// tensor-core shrink skips the same units).
__device__ __forceinline__ bool unit_is_small(int u, const uint32_t *sseg, int nseg, const SegTables &tabs)
{
    if (sseg != nullptr) return (sseg[unit_segment_smem(u, sseg, nseg)] & kSmallBit) != 0;
    return seg_on_warp_shrink(unit_segment(u, tabs), tabs);
}

__device__ __forceinline__ UnitInfo unit_info(int u, const PoolDev &pool, const SegTables &tabs, int T,
                                              int *err, const uint32_t *sseg = nullptr, int nseg = 0)
{
    const int s = sseg != nullptr ? unit_segment_smem(u, sseg, nseg) : unit_segment(u, tabs);
    UnitInfo r;
    r.p0 = tabs.seg_start[s] + (u - tabs.seg_ublk[s]) * kShrinkRows;
    r.p1 = min(r.p0 + kShrinkRows, tabs.seg_start[s + 1]);
    int slot = tabs.seg_slot[s];
#ifdef LORA_CHECK
    // a unit outside the tokens or a slot outside the pool: an empty unit of slot 0
    if (!check_range(r.p0, 0, T, err) || !check_range(r.p1, r.p0, T + 1, err) ||
        !check_range(slot, 0, pool.max_adapters, err)) {
        r.p0 = r.p1 = 0;
        slot = 0;
    }
#endif
    const int32_t *row = pool.slots + (size_t)slot * pool.slot_stride;
    r.npages = row[SLOT_NPAGES];
#ifdef LORA_CHECK
    if (!check_range(r.npages, 1, pool.max_pages + 1, err)) r.npages = 1;
#endif
    r.n = ((r.npages * kRankPage + 15) / 16) * 16;
    r.pages = row + SLOT_PAGES;
    r.scales = row + slot_page_scale(pool.max_pages, 0);
    return r;
}

__global__ void __launch_bounds__(kTcThreads, 1)
    shrink_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmAw,
                     const uint16_t *__restrict__ X, PoolDev pool, SegTables tabs,
                     uint16_t *__restrict__ Vhl, int ldh, int nmax, int stages, uint32_t tmem_cols,
                     int *err, uint64_t *trace, int T, int sseg_cap)
{
    trace_enter_released(trace);
    extern __shared__ uint8_t shrink_smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(shrink_smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t p_bytes = (uint32_t)nmax * 128;  // one box of the A pages
    const uint32_t x_bytes = kSBoxes * kXTileBytes;
    const uint32_t stage_bytes = x_bytes + kSBoxes * p_bytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)stages * stage_bytes);
    uint64_t *empty = full + stages;
    uint64_t *acc_full = empty + stages;  // [2]
    uint64_t *acc_empty = acc_full + 2;   // [2]
    uint64_t *drain = acc_empty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int units = tabs.hdr[HDR_UNITS];
    // the unit prefix and the small flags in shared memory, where they fit: each unit's
    // segment and whether it is skipped then cost no global loads
    const int nseg = tabs.hdr[HDR_NUMSEG];
    uint32_t *sseg = nseg + 1 <= sseg_cap ? tmem_slot + 4 : nullptr;
    if (sseg != nullptr) {
        // four segments a thread per round, every load of a kind issued before any use
        // (the test of seg_on_warp_shrink: rows from `order` only above kShrinkSmallSeg)
        constexpr int kR = 4;
        for (int s0 = threadIdx.x; s0 <= nseg; s0 += kR * (int)blockDim.x) {
            int ub[kR], p0[kR], p1[kR], o0[kR], o1[kR];
#pragma unroll
            for (int j = 0; j < kR; ++j) {
                const int s = s0 + j * (int)blockDim.x;
                ub[j] = s <= nseg ? tabs.seg_ublk[s] : 0;
                p0[j] = s < nseg ? tabs.seg_start[s] : 0;
                p1[j] = s < nseg ? tabs.seg_start[s + 1] : 0;
            }
#pragma unroll
            for (int j = 0; j < kR; ++j) {
                const bool big = p1[j] - p0[j] > kShrinkSmallSeg;
                o0[j] = big ? tabs.order[p0[j]] : 0;
                o1[j] = big ? tabs.order[p1[j] - 1] : 0;
            }
#pragma unroll
            for (int j = 0; j < kR; ++j) {
                const int s = s0 + j * (int)blockDim.x, len = p1[j] - p0[j];
                const bool small = s < nseg && (len <= kShrinkSmallSeg || o1[j] - o0[j] != len - 1);
                if (s <= nseg) sseg[s] = (uint32_t)ub[j] | (small ? kSmallBit : 0u);
            }
        }
    }
    const int d_in = pool.d_in;
    const int KB = (d_in + 64 * kSBoxes - 1) / (64 * kSBoxes);

    if (threadIdx.x == 0) {
        for (int i = 0; i < stages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_empty[i], 4);
        }
        mbar_init(drain, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 5) {
        tmem_alloc(tmem_slot, tmem_cols);
        tmem_relinquish();
    }
    if (warp == 4 && lane == 0) {
        tma_prefetch_map(&tmX);
        tma_prefetch_map(&tmA);
        tma_prefetch_map(&tmAw);
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == 4) {
        // ------------------------------------------------------------ producer
        int it = 0;
        for (int u = blockIdx.x; u < units; u += gridDim.x) {
            if (unit_is_small(u, sseg, nseg, tabs)) continue;  // (every role skips the same units)
            const UnitInfo ui = unit_info(u, pool, tabs, T, err, sseg, nseg);
            const int row0 = LORA_CHECKED(tabs.order[ui.p0], 0, T, err, 0);
            bool contiguous = true;
            for (int r = lane; r < ui.p1 - ui.p0; r += 32)
                contiguous &= (tabs.order[ui.p0 + r] == row0 + r);
            contiguous = __all_sync(0xffffffffu, contiguous);
            const int npad = ui.n / kRankPage;
            // an even number of consecutive pages: one box of nmax rows per 64 columns
            // (rows past the adapter are read but not used by the MMA; past the arena
            // they read as zero) instead of one 1 KB box per page
            bool wide = npad == ui.npages;
            for (int q = 1; q < ui.npages && wide; ++q) wide = ui.pages[q] == ui.pages[0] + q;
            const uint32_t a_bytes = wide ? p_bytes : (uint32_t)npad * 1024u;
            const uint32_t bytes = kSBoxes * (a_bytes + (contiguous ? kXTileBytes : 0u));
            bool ok = true;
            for (int kb = 0; kb < KB && ok; ++kb, ++it) {
                const int s = it % stages;
                const uint32_t ph = (uint32_t)(it / stages) & 1u;
                if (lane == 0) ok = mbar_wait(&empty[s], ph ^ 1u, &abort_flag, err);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                uint8_t *xs = smem + (size_t)s * stage_bytes;
                uint8_t *ps = xs + x_bytes;
                if (!contiguous) {
                    // gather 128 rows x 64 bf16 per box into the 128-byte-swizzled layout;
                    // a row's 16 loads are issued before its stores (a store waiting for
                    // its value would hold up the next load)
                    for (int r = lane; r < 128; r += 32) {
                        const int p = ui.p0 + r;
                        const int tok = (p < ui.p1) ? LORA_CHECKED(tabs.order[p], 0, T, err, -1) : -1;
                        uint4 val[kSBoxes * 8];
#pragma unroll
                        for (int j = 0; j < kSBoxes * 8; ++j) {
                            const int k = kb * kSBoxes * 64 + j * 8;
                            val[j] = make_uint4(0, 0, 0, 0);
                            if (tok >= 0 && k < d_in) val[j] = ldg_nc_v4(X + (size_t)tok * d_in + k);
                        }
#pragma unroll
                        for (int j = 0; j < kSBoxes * 8; ++j) {
                            const int b = j >> 3, c = j & 7;
                            *reinterpret_cast<uint4 *>(xs + b * kXTileBytes + r * 128 + ((c ^ (r & 7)) << 4)) =
                                val[j];
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(&full[s], bytes);
                    for (int b = 0; b < kSBoxes; ++b) {
                        const int k0 = (kb * kSBoxes + b) * 64;
                        if (contiguous) tma_load_2d(xs + b * kXTileBytes, &tmX, &full[s], k0, row0);
                        if (wide) {
                            tma_load_2d(ps + b * p_bytes, &tmAw, &full[s], k0,
                                        LORA_CHECKED(ui.pages[0], 0, pool.num_pages, err, 0) * kRankPage);
                        } else {
                            for (int q = 0; q < npad; ++q) {
                                const int page = q < ui.npages ? LORA_CHECKED(ui.pages[q], 0, pool.num_pages, err, 0) : 0;
                                tma_load_2d(ps + b * p_bytes + q * 1024, &tmA, &full[s], k0,
                                            page * kRankPage);
                            }
                        }
                    }
                }
                __syncwarp();
            }
            if (!ok) break;
        }
        // wait for this CTA's last loads to land before it may exit
        if (lane == 0) {
            for (int i = 0; i < stages && i < it; ++i) {
                const int j = it - 1 - i;
                int dummy = 0;
                mbar_wait(&full[j % stages], (uint32_t)(j / stages) & 1u, &dummy, err);
            }
        }
    } else if (warp == 5) {
        // ----------------------------------------------------------------- MMA
        if (lane == 0) {
            // uc counts the units this CTA runs (not the skipped ones): it picks the
            // accumulator buffer and the phase of its barriers
            int it = 0, uc = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
                if (unit_is_small(u, sseg, nseg, tabs)) continue;
                const UnitInfo ui = unit_info(u, pool, tabs, T, err, sseg, nseg);
                const int buf = uc & 1;
                ok = mbar_wait(&acc_empty[buf], ((uint32_t)(uc >> 1) & 1u) ^ 1u, &abort_flag, err);
                if (!ok) break;
                tc_fence_after_sync();
                const uint32_t idesc = idesc_bf16_f32(128, ui.n);
                const uint32_t d = tmem + (uint32_t)(buf * nmax);
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const int s = it % stages;
                    ok = mbar_wait(&full[s], (uint32_t)(it / stages) & 1u, &abort_flag, err);
                    if (!ok) break;
                    tc_fence_after_sync();
                    const uint32_t xa = smem_u32(smem + (size_t)s * stage_bytes);
                    const uint32_t pa = xa + x_bytes;
#pragma unroll
                    for (int b = 0; b < kSBoxes; ++b)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_bf16_ss(d, sdesc_k_sw128(xa + b * kXTileBytes + kk * 32),
                                        sdesc_k_sw128(pa + b * p_bytes + kk * 32), idesc,
                                        (kb | b | kk) != 0);
                    mma_commit(&empty[s]);
                }
                if (ok) mma_commit(&acc_full[buf]);
                ++uc;
            }
            mma_commit(drain);
            int dummy = 0;
            mbar_wait(drain, 0, &dummy, err);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        int uc = 0;  // units run, as in the MMA role
        for (int u = blockIdx.x; u < units; u += gridDim.x) {
            if (unit_is_small(u, sseg, nseg, tabs)) continue;
            const UnitInfo ui = unit_info(u, pool, tabs, T, err, sseg, nseg);
            const int buf = uc & 1;
            bool ok = true;
            if (lane == 0) ok = mbar_wait(&acc_full[buf], (uint32_t)(uc >> 1) & 1u, &abort_flag, err);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after_sync();
            const int r = warp * 32 + lane;
            const int p = ui.p0 + r;
            const bool valid = p < ui.p1;
            const int tok = valid ? LORA_CHECKED(tabs.order[p], 0, T, err, 0) : 0;
            // s * (X A) as a bf16 pair hi + lo (hi = bf16(v), lo = bf16(v - hi)), grouped
            // per 32 rank columns: [hi 0..31 | lo 0..31] [hi 32..63 | lo 32..63] ...
            uint16_t *hrow = Vhl + (size_t)tok * ldh;
            for (int col = 0; col < ui.n; col += 16) {
                uint32_t v[16];
                tmem_ld16_wait(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(buf * nmax + col), v);
                if (valid) {
                    // each page's columns take that page's scale (a chain's members differ)
                    const float s_lo = __int_as_float(ui.scales[col / kRankPage]);
                    const float s_hi = __int_as_float(ui.scales[col / kRankPage + 1]);
                    uint32_t hi[8], lo[8];
#pragma unroll
                    for (int j = 0; j < 16; j += 2) {
                        const float sc = j < kRankPage ? s_lo : s_hi;
                        const float a0 = sc * __uint_as_float(v[j]);
                        const float a1 = sc * __uint_as_float(v[j + 1]);
                        const uint32_t h = pack_bf16x2(a0, a1);
                        hi[j / 2] = h;
                        lo[j / 2] = pack_bf16x2(a0 - bf16_lo(h), a1 - bf16_hi(h));
                    }
                    uint16_t *dst = hrow + (col / 32) * 64 + (col % 32);
                    *reinterpret_cast<uint4 *>(dst) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                    *reinterpret_cast<uint4 *>(dst + 8) = make_uint4(hi[4], hi[5], hi[6], hi[7]);
                    *reinterpret_cast<uint4 *>(dst + 32) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                    *reinterpret_cast<uint4 *>(dst + 40) = make_uint4(lo[4], lo[5], lo[6], lo[7]);
                }
            }
            if (valid && (ui.n % 32) != 0) {  // the rest of the last 32-column group: zeros
                uint16_t *dst = hrow + (ui.n / 32) * 64 + 16;
                const uint4 z = make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4 *>(dst) = z;
                *reinterpret_cast<uint4 *>(dst + 8) = z;
                *reinterpret_cast<uint4 *>(dst + 32) = z;
                *reinterpret_cast<uint4 *>(dst + 40) = z;
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[buf]);
            ++uc;
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, tmem_cols);
    }
    trace_exit(trace);
}

// ======================================== warp-level shrink of small or scattered segments
//
// One warp per (chunk of up to 16 tokens, page) of the segments seg_on_warp_shrink picks
// (each CTA numbers exactly these work items through a shared-memory prefix of the
// segments' chunk counts; the grid has about a warp per item; each item first requests
// its A page and its X rows into L2 with bulk prefetches):
// D[16 tokens][8 ranks] = X_chunk . A_page^T over d_in with warp-level bf16 MMAs
// (m16n8k16, fp32 accumulation) -- a 16 x 8 tile is what a few tokens of one adapter
// need, far below the tcgen05 tile. The operands come straight from
// global memory in a k order both share (a dot product does not depend on it): in each
// 32-wide step at k0, thread (g = lane / 4, t = lane % 4) loads the 8 inputs k0 + 8t ..
// k0 + 8t + 7 of token rows g and g + 8 and of rank row g of the page, and gives elements
// 0-3 to the first MMA and 4-7 to the second, as the fragment elements of logical columns
// {2t, 2t+1} and {2t+8, 2t+9}. Thread (g, t) ends with D[g][2t..2t+1] and D[g+8][2t..2t+1],
// scales them by the page's scale and writes them in the tensor-core kernel's hi/lo column
// layout (the warp of the adapter's last page also zeroes the rest of its last 32-column
// group).
constexpr int kSmallThreads = 128;
constexpr int kSmallChunk = 16;  // tokens per MMA tile

__device__ __forceinline__ void mma_m16n8k16_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                                  uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__global__ void __launch_bounds__(kSmallThreads)
    shrink_small_kernel(const uint16_t *__restrict__ X, PoolDev pool, SegTables tabs,
                        uint16_t *__restrict__ Vhl, int ldh, int *err, int T, int max_seg)
{
    // in shared memory: the segment starts and, as an exclusive prefix, the number of
    // 16-position chunks of each segment this kernel takes (none for the segments left
    // to the tensor-core shrink), so that the work items are exactly the chunks to do
    extern __shared__ int seg_smem[];
    __shared__ int warp_sum[kSmallThreads / 32];
    const int num_seg = tabs.hdr[HDR_NUMSEG];
    const int nseg = min(num_seg, max_seg);
    int *start = seg_smem, *chk = start + (max_seg + 1);
    for (int s = threadIdx.x; s <= nseg; s += blockDim.x) start[s] = tabs.seg_start[s];
    __syncthreads();
    // each segment's chunk count (0 for a segment left to the tensor-core shrink), from
    // the starts in shared memory: only a segment above kShrinkSmallSeg tokens reads its
    // first and last row from `order` (the test of seg_on_warp_shrink)
    for (int s = threadIdx.x; s < nseg; s += blockDim.x) {
        const int p0 = start[s], len = start[s + 1] - p0;
        const bool mine = len <= kShrinkSmallSeg || tabs.order[p0 + len - 1] - tabs.order[p0] != len - 1;
        chk[s] = mine ? (len + kSmallChunk - 1) / kSmallChunk : 0;
    }
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, g = lane >> 2, t = lane & 3;
    {
        // each thread a contiguous run of segments: its count, a scan across the block,
        // then the run's prefixes (in place of the counts)
        const int per = (nseg + kSmallThreads - 1) / kSmallThreads;
        const int s0 = min(nseg, (int)threadIdx.x * per), s1 = min(nseg, s0 + per);
        int local = 0;
        for (int s = s0; s < s1; ++s) local += chk[s];
        int incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) warp_sum[warp] = incl;
        __syncthreads();
        int base = 0, total = 0;
#pragma unroll
        for (int w = 0; w < kSmallThreads / 32; ++w) {
            if (w < warp) base += warp_sum[w];
            total += warp_sum[w];
        }
        int run = base + incl - local;
        for (int s = s0; s < s1; ++s) {
            const int n = chk[s];
            chk[s] = run;
            run += n;
        }
        if (threadIdx.x == 0) chk[nseg] = total;
        __syncthreads();
    }
    const int gw = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    const int nw = (int)((gridDim.x * blockDim.x) >> 5);
    const int P = pool.max_pages, d_in = pool.d_in;
    // work items (chunk, page) in segment order: the grid has about a warp per item
    const int items = chk[nseg] * P;
    for (int v = gw; v < items; v += nw) {
        const int c = v / P, q = v - c * P;
        int lo = 0, hi = nseg;  // the chunk's segment: the largest s with chk[s] <= c
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (chk[mid] <= c) lo = mid; else hi = mid;
        }
        const int s = lo;
        const int p0 = start[s] + (c - chk[s]) * kSmallChunk;
        const int p1u = start[s + 1];
        if (p0 >= p1u) continue;
        const int len = min(kSmallChunk, p1u - p0);
#ifdef LORA_CHECK
        if (!check_range(p0, 0, T, err) || !check_range(p0 + len, p0, T + 1, err)) continue;
#endif
        const int slot = LORA_CHECKED(tabs.seg_slot[s], 0, pool.max_adapters, err, 0);
        const int32_t *row = pool.slots + (size_t)slot * pool.slot_stride;
        const int npages = row[SLOT_NPAGES];
        if (q >= npages) continue;
        const int page = LORA_CHECKED(row[SLOT_PAGES + q], 0, pool.num_pages, err, 0);
        const float scale = __int_as_float(row[slot_page_scale(P, q)]);
        const bool has0 = g < len, has8 = g + 8 < len;
        const int tok0 = has0 ? LORA_CHECKED(tabs.order[p0 + g], 0, T, err, 0) : 0;
        const int tok8 = has8 ? LORA_CHECKED(tabs.order[p0 + g + 8], 0, T, err, 0) : 0;
        // the page (8 rows of d_in, contiguous) and the chunk's X rows requested into L2 as
        // whole rows, so the rounds of loads below hit L2 instead of trickling from DRAM
        if (lane == 0) prefetch_l2_bulk(pool.A_pages + (size_t)page * kRankPage * d_in, (uint32_t)(kRankPage * d_in * 2));
        if (t == 0 && has0) prefetch_l2_bulk(X + (size_t)tok0 * d_in, (uint32_t)(d_in * 2));
        if (t == 0 && has8) prefetch_l2_bulk(X + (size_t)tok8 * d_in, (uint32_t)(d_in * 2));
        const uint16_t *x0 = X + (size_t)tok0 * d_in + 8 * t;
        const uint16_t *x8 = X + (size_t)tok8 * d_in + 8 * t;
        const uint16_t *ar = pool.A_pages + ((size_t)page * kRankPage + g) * d_in + 8 * t;
        float d[4] = {0.f, 0.f, 0.f, 0.f}, e[4] = {0.f, 0.f, 0.f, 0.f};
        const uint4 z = make_uint4(0, 0, 0, 0);
        // eight 32-wide steps per round: all their loads are issued before their MMAs
        // (the loads and the MMAs are asm statements that keep their program order)
        constexpr int kSteps = 8;
        for (int k0 = 0; k0 < d_in; k0 += 32 * kSteps) {
            uint4 xa[kSteps], xb[kSteps], w[kSteps];
#pragma unroll
            for (int j = 0; j < kSteps; ++j) {
                const int k = k0 + 32 * j;
                const bool in = k + 8 * t < d_in;  // d_in is a multiple of 8
                xa[j] = has0 && in ? ldg_nc_v4(x0 + k) : z;
                xb[j] = has8 && in ? ldg_nc_v4(x8 + k) : z;
                w[j] = in ? ldg_nc_v4(ar + k) : z;
            }
#pragma unroll
            for (int j = 0; j < kSteps; ++j) {
                mma_m16n8k16_bf16(d, xa[j].x, xb[j].x, xa[j].y, xb[j].y, w[j].x, w[j].y);
                mma_m16n8k16_bf16(e, xa[j].z, xb[j].z, xa[j].w, xb[j].w, w[j].z, w[j].w);
            }
        }
        // token g: ranks 2t, 2t+1 in d[0..1] + e[0..1]; token g + 8: in d[2..3] + e[2..3]
        const int col = q * kRankPage + 2 * t;
        const int group_end = ((npages * kRankPage + 31) / 32) * 32;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            if (half == 0 ? !has0 : !has8) continue;
            const float a0 = scale * (d[2 * half] + e[2 * half]);
            const float a1 = scale * (d[2 * half + 1] + e[2 * half + 1]);
            const uint32_t hv = pack_bf16x2(a0, a1);
            const uint32_t lv = pack_bf16x2(a0 - bf16_lo(hv), a1 - bf16_hi(hv));
            uint16_t *hrow = Vhl + (size_t)(half == 0 ? tok0 : tok8) * ldh;
            uint16_t *dst = hrow + (col / 32) * 64 + (col % 32);
            *reinterpret_cast<uint32_t *>(dst) = hv;
            *reinterpret_cast<uint32_t *>(dst + 32) = lv;
            if (q == npages - 1)  // the rest of the last 32-column group: zeros
                for (int zc = q * kRankPage + kRankPage + 2 * t; zc < group_end; zc += 8) {
                    uint16_t *zd = hrow + (zc / 32) * 64 + (zc % 32);
                    *reinterpret_cast<uint32_t *>(zd) = 0u;
                    *reinterpret_cast<uint32_t *>(zd + 32) = 0u;
                }
        }
    }
}

uint32_t pow2_cols(uint32_t n)
{
    uint32_t c = 32;
    while (c < n) c <<= 1;
    return c;
}

}  // namespace

cudaError_t launch_shrink_small(const uint16_t *X, int T, const PoolDev &pool, SegTables tabs, uint16_t *Vhl,
                                int ldh, int num_sms, int *err, cudaStream_t stream)
{
    // the segment tables of up to min(T, adapters) segments in shared memory
    const int max_seg = T < pool.max_adapters ? T : pool.max_adapters;
    const size_t smem = 2 * ((size_t)max_seg + 1) * sizeof(int);
    cudaError_t e = ensure_smem_attr((const void *)shrink_small_kernel, smem);
    if (e != cudaSuccess) return e;
    // about a warp per work item (chunk, page): up to T / 16 + segments chunks
    const long long max_items = ((long long)T / kSmallChunk + max_seg) * pool.max_pages;
    const long long want = (max_items + kSmallThreads / 32 - 1) / (kSmallThreads / 32);
    const int grid = (int)std::max<long long>(num_sms, std::min<long long>(want, 8ll * num_sms));
    shrink_small_kernel<<<grid, kSmallThreads, smem, stream>>>(X, pool, tabs, Vhl, ldh, err, T, max_seg);
    return cudaGetLastError();
}

cudaError_t launch_shrink_tc(const CUtensorMap &tmX, const CUtensorMap &tmA,
                             const CUtensorMap &tmAw, const uint16_t *X,
                             int T, const PoolDev &pool, SegTables tabs, uint16_t *Vhl, int ldh,
                             int num_sms, int *err, cudaStream_t stream, uint64_t *trace)
{
    const int nmax = ((pool.max_pages * kRankPage + 15) / 16) * 16;
    const size_t stage_bytes = kSBoxes * (kXTileBytes + (size_t)nmax * 128);
    int stages = (int)((200 * 1024) / stage_bytes);
    if (stages > 6) stages = 6;
    if (stages < 2) stages = 2;
    const int max_seg = T < pool.max_adapters ? T : pool.max_adapters;
    // the segments' unit prefix in shared memory when it fits in 16 KB
    const int sseg_cap = max_seg + 1 <= 4096 ? max_seg + 1 : 0;
    const size_t smem = 1024 + stages * stage_bytes + (2 * stages + 5) * 8 + 16 + (size_t)sseg_cap * 4;
    const uint32_t tmem_cols = pow2_cols(2 * nmax);
    const int max_units = (T + kShrinkRows - 1) / kShrinkRows + max_seg;
    int grid = max_units < num_sms ? max_units : num_sms;
    if (grid <= 0) return cudaSuccess;
    cudaError_t e = ensure_smem_attr((const void *)shrink_tc_kernel, smem);
    if (e != cudaSuccess) return e;
    shrink_tc_kernel<<<grid, kTcThreads, smem, stream>>>(tmX, tmA, tmAw, X, pool, tabs, Vhl, ldh, nmax,
                                                          stages, tmem_cols, err, trace, T, sseg_cap);
    return cudaGetLastError();
}

}  // namespace lora
