// gemm_decode.cu -- the decode path (T <= 256): two kernels per call, for one
// layer or for a group of layers that share the token ids (e.g. the target
// modules of one transformer layer), described by one problem table.
//
// 1. gemm_decode_kernel: base products + the per-token low-rank shrink.
//    At decode sizes the base GEMM is bound by reading W_base once from HBM, so
//    the layout is chosen to stream W at full bandwidth on every SM:
//    * operands swapped: D[n, t] = sum_k W[n,k] X[t,k], so the long d_out side
//      is the MMA's M (128 rows of W per tile) and the T tokens are its N
//      (T rounded up to 16; rows past T read as zero from TMA);
//    * stream-K: the problems' (tile, 128-wide k-block) units, concatenated in
//      problem order, are cut into G equal contiguous ranges, one per CTA
//      (G = number of SMs, or fewer for small problems; small layers launch
//      extra CTAs that only take shrink pairs), so every SM streams
//      the same share of all the weights of the group. Every tile a range
//      touches (a "segment" of the range) gets a TMEM accumulator from a small
//      ring and is written out as an fp32 partial sum [cta][segment][T][128];
//    * warp roles: warp 4 issues TMA loads (per stage two W boxes 128x64 and two
//      X boxes T'x64, 128-byte swizzle) into a multi-stage ring -- the first
//      ring's worth of W (a weight) before the wait on the previous kernel;
//      warp 5 allocates TMEM and issues tcgen05 MMAs (M=128, N=T', K=16);
//      warps 0-3, idle until the accumulators are ready, first compute the
//      low-rank shrink V[t, 8q..8q+7] = s_i X[t,:] A_i[:, 8q..8q+7] for the
//      (problem, token, page) triples dealt to this CTA round-robin (a
//      BGMV-style per-token gather: each reads one 8 x d_in A page with 128-bit
//      loads; one pair at a time on all four warps, or, when a CTA has several,
//      one pair per warp), so the adapter reads overlap the W stream; then they read the
//      accumulators back with tcgen05.ld (TMEM lane = output row n) and store
//      the partials.
// 2. finish_decode_kernel (launched with programmatic stream serialization, so
//    it is resident and has loaded its B pages before the GEMM ends): per
//    output element, the partials of the CTAs that covered its tile are summed
//    in CTA order (deterministic), the low-rank expand s_i V[t,:] B_i[:,n] is
//    added from the interleaved B pages (one 16-byte load = 8 rank rows of one
//    column; V already carries s_i), and the sum is rounded once to bf16.
#include <algorithm>
#include <utility>

#include "device_common.cuh"

namespace lora {

namespace {

constexpr int kThreads = 192;
constexpr int kWTileBytes = 128 * 128;  // one TMA box of W: 128 rows x 64 bf16
// Two 64-wide boxes per stage (k-block = 128 columns): half the barrier round
// trips per byte and longer runs per W row than one box, measured ~2.5 us
// faster per q_proj decode step; four boxes were no faster.
constexpr int kBoxes = 2;
constexpr uint32_t kBarSetup = 1;       // named barrier: all six warps, setup done
constexpr uint32_t kBarShrink = 2;      // named barrier: the four epilogue warps

__host__ __device__ __forceinline__ int cta_start(int c, int U, int G)
{
    return (int)(((long long)c * U) / G);
}

// Index into a plan's problem table: a compile-time 0 for a one-problem plan, so
// its fields are read at fixed parameter offsets.
template <int NP>
__host__ __device__ __forceinline__ int pick(int m)
{
    return NP == 1 ? 0 : m;
}

// The problem that unit u belongs to: the last m whose first unit is <= u.
template <class Plan>
__host__ __device__ __forceinline__ int unit_problem(const Plan &p, int u)
{
    if (Plan::kNP == 1) return 0;
    int m = 0;
    for (int k = 1; k < p.n; ++k)
        if (p.prob[k].u_begin <= u) m = k;
    return m;
}

// Index of unit u's tile in the problems' concatenated tile order.
template <class Plan>
__host__ __device__ __forceinline__ int unit_tile(const Plan &p, int u)
{
    const DecodeProblem &q = p.prob[pick<Plan::kNP>(unit_problem(p, u))];
    return q.g_begin + (u - q.u_begin) / q.KB;
}

// One (token, page) pair of the shrink, computed by the 128 threads of warps 0-3.
// UNR: chunks of d_in whose loads one thread has in flight at a time (the shrink is
// bound by the loads in flight per SM; the register-bounded kernel variant keeps 2).
template <int UNR>
__device__ __forceinline__ void shrink_pair(int t, int page, float scale, const DecodeProblem &pr,
                                            int q, float (*red)[8])
{
    const int tid = threadIdx.x;  // 0..127
    const int warp = tid >> 5, lane = tid & 31;
    const int d_in = pr.pool.d_in;
    const uint16_t *Ap = pr.pool.A_pages + (size_t)page * kRankPage * d_in;
    const uint16_t *xr = pr.X + (size_t)t * d_in;
    float acc[kRankPage];
#pragma unroll
    for (int jj = 0; jj < kRankPage; ++jj) acc[jj] = 0.f;
#pragma unroll UNR
    for (int c = tid; c < d_in / 8; c += 128) {
        const uint4 x = ldg_nc_v4(xr + c * 8);
        uint4 a[kRankPage];
#pragma unroll
        for (int jj = 0; jj < kRankPage; ++jj) a[jj] = ldg_nc_v4(Ap + (size_t)jj * d_in + c * 8);
#pragma unroll
        for (int jj = 0; jj < kRankPage; ++jj) acc[jj] = dot8_bf16(x, a[jj], acc[jj]);
    }
#pragma unroll
    for (int jj = 0; jj < kRankPage; ++jj)
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) acc[jj] += __shfl_xor_sync(0xffffffffu, acc[jj], o);
    if (lane == 0)
#pragma unroll
        for (int jj = 0; jj < kRankPage; ++jj) red[warp][jj] = acc[jj];
    named_bar_sync(kBarShrink, 128);
    if (tid < kRankPage) {
        const float s = red[0][tid] + red[1][tid] + red[2][tid] + red[3][tid];
        pr.V[(size_t)t * pr.ldv + q * kRankPage + tid] = scale * s;
    }
    named_bar_sync(kBarShrink, 128);
}

// The same pair computed by one warp alone (lanes stride over d_in): when a CTA has
// several pairs, its four epilogue warps each take one and run them in parallel.
template <int UNR>
__device__ __forceinline__ void shrink_pair_warp(int t, int page, float scale, const DecodeProblem &pr,
                                                 int q)
{
    const int lane = threadIdx.x & 31;
    const int d_in = pr.pool.d_in;
    const uint16_t *Ap = pr.pool.A_pages + (size_t)page * kRankPage * d_in;
    const uint16_t *xr = pr.X + (size_t)t * d_in;
    float acc[kRankPage];
#pragma unroll
    for (int jj = 0; jj < kRankPage; ++jj) acc[jj] = 0.f;
#pragma unroll UNR
    for (int c = lane; c < d_in / 8; c += 32) {
        const uint4 x = ldg_nc_v4(xr + c * 8);
        uint4 a[kRankPage];
#pragma unroll
        for (int jj = 0; jj < kRankPage; ++jj) a[jj] = ldg_nc_v4(Ap + (size_t)jj * d_in + c * 8);
#pragma unroll
        for (int jj = 0; jj < kRankPage; ++jj) acc[jj] = dot8_bf16(x, a[jj], acc[jj]);
    }
    float mine = 0.f;
#pragma unroll
    for (int jj = 0; jj < kRankPage; ++jj) {
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) acc[jj] += __shfl_xor_sync(0xffffffffu, acc[jj], o);
        if (lane == jj) mine = acc[jj];
    }
    if (lane < kRankPage) pr.V[(size_t)t * pr.ldv + q * kRankPage + lane] = scale * mine;
}

// The current problem's unit bookkeeping, kept in registers while a loop walks
// its units in order (reloaded when the walk crosses into the next problem).
struct UnitCursor {
    int m, ub, KB, gb, next_ub;
    template <class Plan>
    __device__ __forceinline__ void load(const Plan &p, int mm)
    {
        m = pick<Plan::kNP>(mm);
        const DecodeProblem &q = p.prob[m];
        ub = q.u_begin;
        KB = q.KB;
        gb = q.g_begin;
        next_ub = Plan::kNP > 1 && m + 1 < p.n ? p.prob[pick<Plan::kNP>(m + 1)].u_begin : 0x7fffffff;
    }
    template <class Plan>
    __device__ __forceinline__ void seek(const Plan &p, int u)
    {
        while (u >= next_ub) load(p, m + 1);
    }
};

// Warps 0-3 of a decode GEMM kernel (either base format): after the setup barrier
// over `threads` threads, the shrink pairs dealt to this CTA (after the wait on the
// previous kernel), then each of its segments' accumulators read out of TMEM into the
// split-K partial sums.
template <int NP, int UNR = 2>
__device__ __forceinline__ void decode_epilogue(const DecodePlanT<NP> &p, const int32_t *__restrict__ ids,
                                                float *__restrict__ partials, int *err, int c, int nseg,
                                                uint64_t *acc_full, uint64_t *acc_empty,
                                                volatile int *abort_flag_p, float (*red)[kRankPage],
                                                const uint32_t *tmem_slot, uint32_t threads)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_acc = p.n_acc;
    named_bar_sync(kBarSetup, threads);
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    // Before the wait on the previous kernel: the A pages of this CTA's shrink pairs
    // into L2, one bulk prefetch per page (a thread per pair), so the per-lane loads
    // of the shrink below hit L2. The ids read here may still be written by an
    // earlier kernel in the stream, so they only steer these requests; the pairs
    // below read the ids again after the wait.
    if (ids != nullptr && p.prefetch_a) {
        int m = 0;
        for (int u = c + (int)threadIdx.x * (int)gridDim.x; u < p.pairs; u += 128 * (int)gridDim.x) {
            while (NP > 1 && m + 1 < p.n && p.prob[pick<NP>(m + 1)].pair_begin <= u) ++m;
            const DecodeProblem &pr = p.prob[pick<NP>(m)];
            const int lp = u - pr.pair_begin;
            const int t = lp / pr.pool.max_pages, q = lp - t * pr.pool.max_pages;
            const int id = ids[t];
            if (!slot_loaded(pr.pool.slots, pr.pool.slot_stride, pr.pool.max_adapters, id)) continue;
            const int32_t *row = pr.pool.slots + (size_t)id * pr.pool.slot_stride;
            if (q >= row[SLOT_NPAGES]) continue;
            const int page = row[SLOT_PAGES + q];
            if (page < 0 || page >= pr.pool.num_pages) continue;
            prefetch_l2_bulk(pr.pool.A_pages + (size_t)page * kRankPage * pr.pool.d_in,
                             (uint32_t)(kRankPage * pr.pool.d_in * 2));
        }
    }
    pdl_wait_prior();  // X, ids, V and the partials belong to the stream's order
    if (ids != nullptr) {
        // this CTA's pairs: c, c + grid, c + 2 grid, ...; with more than one of them
        // on average the four warps take every fourth pair each, else all 128
        // threads work on one pair at a time
        const int stride = (int)gridDim.x;
        const bool by_warp = p.pairs > stride;
        int m = 0;
        for (int u = by_warp ? c + warp * stride : c; u < p.pairs; u += by_warp ? 4 * stride : stride) {
            while (NP > 1 && m + 1 < p.n && p.prob[pick<NP>(m + 1)].pair_begin <= u) ++m;
            const DecodeProblem &pr = p.prob[pick<NP>(m)];
            const int lp = u - pr.pair_begin;
            const int t = lp / pr.pool.max_pages, q = lp - t * pr.pool.max_pages;
            const int id = ids[t];
            if (!slot_loaded(pr.pool.slots, pr.pool.slot_stride, pr.pool.max_adapters, id)) continue;
            const int32_t *row = pr.pool.slots + (size_t)id * pr.pool.slot_stride;
            if (q >= row[SLOT_NPAGES]) continue;
            const float scale = __int_as_float(row[slot_page_scale(pr.pool.max_pages, q)]);
            const int page = LORA_CHECKED(row[SLOT_PAGES + q], 0, pr.pool.num_pages, pr.err, 0);
            if (by_warp)
                shrink_pair_warp<UNR>(t, page, scale, pr, q);
            else
                shrink_pair<UNR>(t, page, scale, pr, q, red);
        }
    }
    for (int seg = 0; seg < nseg; ++seg) {
#ifdef LORA_CHECK
        if (!check_range(seg, 0, p.max_seg, err)) break;
#endif
        const int a = seg % n_acc;
        bool ok = true;
        if (lane == 0) ok = mbar_wait(&acc_full[a], (uint32_t)(seg / n_acc) & 1u, abort_flag_p, err);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        tc_fence_after_sync();
        float *out = partials + ((size_t)c * p.max_seg + seg) * p.T * 128 + warp * 32 + lane;
        for (int col = 0; col < p.ntok; col += 16) {
            uint32_t v[16];
            tmem_ld16_wait(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(a * p.ntok + col), v);
#pragma unroll
            for (int j = 0; j < 16; ++j)
                if (col + j < p.T) out[(size_t)(col + j) * 128] = __uint_as_float(v[j]);
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[a]);
    }
}

template <int NP, int UNR = 2>
__device__ __forceinline__ void gemm_decode_body(const DecodeMapsT<NP> &maps, const DecodePlanT<NP> &p,
                                                 const int32_t *__restrict__ ids,
                                                 float *__restrict__ partials, int *err)
{
    extern __shared__ uint8_t dec_smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(dec_smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t x_box = (uint32_t)p.ntok * 128;  // one TMA box of X
    const uint32_t w_bytes = kBoxes * kWTileBytes;
    const uint32_t stage_bytes = w_bytes + kBoxes * x_box;
    const int stages = p.stages, n_acc = p.n_acc;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)stages * stage_bytes);
    uint64_t *empty = full + stages;
    uint64_t *acc_full = empty + stages;     // [n_acc]
    uint64_t *acc_empty = acc_full + n_acc;  // [n_acc]
    uint64_t *drain = acc_empty + n_acc;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    __shared__ int abort_flag;
    __shared__ float red[4][kRankPage];

    // the finishing kernel may start its independent prologue now
    pdl_launch_dependents();
    uint64_t *const trace = p.trace ? p.trace + 2 * kTraceWords : nullptr;  // kernel slot 2
    trace_enter(trace);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.x;
    // CTAs past the G stream-K ranges (launched when the shrink has more pairs than
    // there are ranges) only run shrink pairs
    const bool ranged = c < p.G;
    const int u0 = ranged ? cta_start(c, p.U, p.G) : 0, u1 = ranged ? cta_start(c + 1, p.U, p.G) : 0;
    const int g0 = unit_tile(p, u0);  // the tile of segment 0
    const int nseg = u1 > u0 ? unit_tile(p, u1 - 1) - g0 + 1 : 0;

    if (warp == 4) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            for (int i = 0; i < stages; ++i) {
                mbar_init(&full[i], 1);
                mbar_init(&empty[i], 1);
            }
            for (int i = 0; i < n_acc; ++i) {
                mbar_init(&acc_full[i], 1);
                mbar_init(&acc_empty[i], 4);
            }
            mbar_init(drain, 1);
            abort_flag = 0;
            fence_mbar_init();
            for (int m = 0; m < p.n; ++m) {
                tma_prefetch_map(&maps.W[m]);
                tma_prefetch_map(&maps.X[m]);
            }
        }
        __syncwarp();
        named_bar_arrive(kBarSetup, kThreads);  // barriers are ready; do not wait for TMEM
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();  // W is read exactly once
            // W is a weight: the first ring's worth of W tiles is requested before the
            // previous kernel in the stream has finished; X (and everything the epilogue
            // touches) only after the programmatic wait.
            const int pre = (u1 - u0) < stages ? (u1 - u0) : stages;
            UnitCursor cur;
            cur.load(p, unit_problem(p, u0));
            for (int i = 0; i < pre; ++i) {
                const int u = u0 + i;
                cur.seek(p, u);
                const int lu = u - cur.ub, tile = lu / cur.KB, kb = lu - tile * cur.KB;
                mbar_arrive_expect_tx(&full[i], stage_bytes);
                for (int b = 0; b < kBoxes; ++b)
                    tma_load_2d_hint(smem + (size_t)i * stage_bytes + b * kWTileBytes, &maps.W[cur.m],
                                     &full[i], (kb * kBoxes + b) * 64, tile * 128, pol_w);
            }
            pdl_wait_prior();
            trace_release(trace);
            cur.load(p, unit_problem(p, u0));
            for (int i = 0; i < pre; ++i) {
                const int u = u0 + i;
                cur.seek(p, u);
                const int kb = (u - cur.ub) % cur.KB;
                for (int b = 0; b < kBoxes; ++b)
                    tma_load_2d(smem + (size_t)i * stage_bytes + w_bytes + b * x_box, &maps.X[cur.m],
                                &full[i], (kb * kBoxes + b) * 64, 0);
            }
            int it = pre;
            for (int u = u0 + pre; u < u1; ++u, ++it) {
                const int s = it % stages;
                if (!mbar_wait(&empty[s], ((uint32_t)(it / stages) & 1u) ^ 1u, &abort_flag, err)) break;
                cur.seek(p, u);
                const int lu = u - cur.ub, tile = lu / cur.KB, kb = lu - tile * cur.KB;
                uint8_t *ws = smem + (size_t)s * stage_bytes;
                mbar_arrive_expect_tx(&full[s], stage_bytes);
                for (int b = 0; b < kBoxes; ++b) {
                    tma_load_2d_hint(ws + b * kWTileBytes, &maps.W[cur.m], &full[s],
                                     (kb * kBoxes + b) * 64, tile * 128, pol_w);
                    tma_load_2d(ws + w_bytes + b * x_box, &maps.X[cur.m], &full[s],
                                (kb * kBoxes + b) * 64, 0);
                }
            }
            // do not leave while copies into this CTA's shared memory are in flight
            for (int i = 0; i < stages && i < it; ++i) {
                const int j = it - 1 - i;
                int dummy = 0;
                mbar_wait(&full[j % stages], (uint32_t)(j / stages) & 1u, &dummy, err);
            }
        }
        __syncwarp();
    } else if (warp == 5) {
        // ----------------------------------------------------------------- MMA
        tmem_alloc(tmem_slot, p.tmem_cols);
        tmem_relinquish();
        tc_fence_before_sync();
        named_bar_sync(kBarSetup, kThreads);
        tc_fence_after_sync();
        const uint32_t tmem = *tmem_slot;
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(128, p.ntok);
            int it = 0;
            UnitCursor cur;
            cur.load(p, unit_problem(p, u0));
            uint32_t d = tmem;
            for (int u = u0; u < u1; ++u, ++it) {
                cur.seek(p, u);
                const int KB = cur.KB, lu = u - cur.ub;
                const int tile = lu / KB, kb = lu - tile * KB;
                const int seg = cur.gb + tile - g0;
                const bool seg_first = (kb == 0) || (u == u0);
                if (seg_first) {
                    // the ring slot's previous tile must have been read out
                    const int a = seg % n_acc;
                    if (!mbar_wait(&acc_empty[a], ((uint32_t)(seg / n_acc) & 1u) ^ 1u, &abort_flag, err))
                        break;
                    tc_fence_after_sync();
                    d = tmem + (uint32_t)(a * p.ntok);
                }
                const int s = it % stages;
                if (!mbar_wait(&full[s], (uint32_t)(it / stages) & 1u, &abort_flag, err)) break;
                tc_fence_after_sync();
                const uint32_t wa = smem_u32(smem + (size_t)s * stage_bytes);
                const uint32_t xa = wa + w_bytes;
#pragma unroll
                for (int b = 0; b < kBoxes; ++b)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_bf16_ss(d, sdesc_k_sw128(wa + b * kWTileBytes + kk * 32),
                                    sdesc_k_sw128(xa + b * x_box + kk * 32), idesc,
                                    (seg_first && b == 0 && kk == 0) ? 0u : 1u);
                mma_commit(&empty[s]);
                if (u == u1 - 1 || kb == KB - 1) mma_commit(&acc_full[seg % n_acc]);
            }
            mma_commit(drain);
            int dummy = 0;
            mbar_wait(drain, 0, &dummy, err);
        }
        __syncwarp();
    } else {
        // ------------------------------------- warps 0-3: shrink, then epilogue
        decode_epilogue<NP, UNR>(p, ids, partials, err, c, nseg, acc_full, acc_empty, &abort_flag, red, tmem_slot,
                            kThreads);
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after_sync();
        tmem_dealloc(*tmem_slot, p.tmem_cols);
    }
    trace_exit(trace);
}

// ------------------------------------------------------------- 4-bit base
//
// gemm_decode_q4_kernel: the same stream-K split, accumulator ring, shrink and split-K
// partial sums as gemm_decode_kernel (one layer), for a base stored as 4-bit codes
// with one bf16 scale and one 4-bit zero point per (group of 128 inputs, output row):
// W = bf16(s (q - z)). W is a quarter of the bytes, and the MMA still takes bf16, so
// the tiles are dequantised in shared memory:
//  * warp 4 streams the codes of each (tile, k-block) unit (128 rows x 64 bytes) with
//    its 128 scales and zero points into a deep ring of 9 KB stages; they are weights,
//    so nothing waits on the previous kernel;
//  * warps 7-10 turn a unit's codes into the bf16 W tile of an operand stage, in the
//    128-byte-swizzled layout a TMA load would have written: one thread per W row, its
//    64 code bytes read as four 16-byte words issued together (in an order rotated by
//    lane pair, so that 8 lanes touch 8 different bank groups), 8 values per 4 bytes by
//    dequant8_q4, stored as 16 chunks (conflict-free through the swizzle);
//  * warp 6 loads X into the same operand stage after the wait on the previous kernel;
//    the stage is full when its X bytes have landed and the four dequant warps have
//    arrived;
//  * warp 5 issues the MMAs exactly as for a bf16 base; warps 0-3 as there.
// The first operand stages are dequantised before the previous kernel ends.
constexpr int kQ4Threads = 352;
constexpr int kQ4CodeBytes = 128 * 64;          // one unit's codes
constexpr int kQ4RawBytes = 9216;               // codes + 128 scales + 128 zero points, 1 KB aligned

__device__ __forceinline__ void gemm_decode_q4_body(const DecodeMapsQ4 &maps, const DecodePlanT<1> &p,
                                                    const int32_t *__restrict__ ids,
                                                    float *__restrict__ partials, int *err)
{
    extern __shared__ uint8_t dec_smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(dec_smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t x_box = (uint32_t)p.ntok * 128;
    const uint32_t w_bytes = kBoxes * kWTileBytes;
    const uint32_t stage_bytes = w_bytes + kBoxes * x_box;
    const int stages = p.stages, raw = p.raw_stages, n_acc = p.n_acc;
    uint8_t *rawbuf = smem + (size_t)stages * stage_bytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(rawbuf + (size_t)raw * kQ4RawBytes);
    uint64_t *empty = full + stages;
    uint64_t *raw_full = empty + stages;     // [raw]
    uint64_t *raw_empty = raw_full + raw;    // [raw]
    uint64_t *acc_full = raw_empty + raw;    // [n_acc]
    uint64_t *acc_empty = acc_full + n_acc;  // [n_acc]
    uint64_t *drain = acc_empty + n_acc;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    __shared__ int abort_flag;
    __shared__ float red[4][kRankPage];

    pdl_launch_dependents();  // the finishing kernel reads nothing before its own wait
    uint64_t *const trace = p.trace ? p.trace + 2 * kTraceWords : nullptr;  // kernel slot 2
    trace_enter(trace);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.x;
    const bool ranged = c < p.G;
    const int u0 = ranged ? cta_start(c, p.U, p.G) : 0, u1 = ranged ? cta_start(c + 1, p.U, p.G) : 0;
    const int KB = p.prob[0].KB;
    const int g0 = u0 / KB;
    const int nseg = u1 > u0 ? (u1 - 1) / KB - g0 + 1 : 0;

    if (warp == 4) {
        // ------------------------------------------------------- codes producer
        if (lane == 0) {
            for (int i = 0; i < stages; ++i) {
                mbar_init(&full[i], 1 + 4);  // X producer (with its bytes) + four dequant warps
                mbar_init(&empty[i], 1);
            }
            for (int i = 0; i < raw; ++i) {
                mbar_init(&raw_full[i], 1);
                mbar_init(&raw_empty[i], 4);
            }
            for (int i = 0; i < n_acc; ++i) {
                mbar_init(&acc_full[i], 1);
                mbar_init(&acc_empty[i], 4);
            }
            mbar_init(drain, 1);
            abort_flag = 0;
            fence_mbar_init();
            tma_prefetch_map(&maps.Wq);
            tma_prefetch_map(&maps.S);
            tma_prefetch_map(&maps.Z);
            tma_prefetch_map(&maps.X);
        }
        __syncwarp();
        named_bar_arrive(kBarSetup, kQ4Threads);
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();  // read exactly once
            int it = 0;
            for (int u = u0; u < u1; ++u, ++it) {
                const int i = it % raw;
                if (it >= raw && !mbar_wait_inl(&raw_empty[i], ((uint32_t)(it / raw) & 1u) ^ 1u, &abort_flag, err))
                    break;
                const int tile = u / KB, kb = u - tile * KB;
                uint8_t *rb = rawbuf + (size_t)i * kQ4RawBytes;
                mbar_arrive_expect_tx(&raw_full[i], kQ4CodeBytes + 128 * 2 + 128);
                tma_load_2d_hint(rb, &maps.Wq, &raw_full[i], kb * 64, tile * 128, pol);
                tma_load_2d(rb + kQ4CodeBytes, &maps.S, &raw_full[i], tile * 128, kb);
                tma_load_2d(rb + kQ4CodeBytes + 256, &maps.Z, &raw_full[i], tile * 128, kb);
            }
            for (int i = 0; i < raw && i < it; ++i) {  // no exit while copies are in flight
                const int j = it - 1 - i;
                int dummy = 0;
                mbar_wait(&raw_full[j % raw], (uint32_t)(j / raw) & 1u, &dummy, err);
            }
        }
        __syncwarp();
    } else if (warp == 6) {
        // ----------------------------------------------------------- X producer
        named_bar_sync(kBarSetup, kQ4Threads);
        if (lane == 0) {
            pdl_wait_prior();  // X belongs to the stream's order
            trace_release(trace);
            int it = 0;
            for (int u = u0; u < u1; ++u, ++it) {
                const int st = it % stages;
                if (it >= stages &&
                    !mbar_wait_inl(&empty[st], ((uint32_t)(it / stages) & 1u) ^ 1u, &abort_flag, err))
                    break;
                const int kb = u % KB;
                uint8_t *xs = smem + (size_t)st * stage_bytes + w_bytes;
                mbar_arrive_expect_tx(&full[st], kBoxes * x_box);
                for (int b = 0; b < kBoxes; ++b)
                    tma_load_2d(xs + b * x_box, &maps.X, &full[st], (kb * kBoxes + b) * 64, 0);
            }
            for (int i = 0; i < stages && i < it; ++i) {
                const int j = it - 1 - i;
                int dummy = 0;
                mbar_wait(&full[j % stages], (uint32_t)(j / stages) & 1u, &dummy, err);
            }
        }
        __syncwarp();
    } else if (warp >= 7) {
        // ------------------------------------------------------- dequant warps
        named_bar_sync(kBarSetup, kQ4Threads);
        const int row = (warp - 7) * 32 + lane;  // this thread's W row of each tile
        const int rot = (lane >> 1) & 3;
        int it = 0;
        for (int u = u0; u < u1; ++u, ++it) {
            const int i = it % raw, st = it % stages;
            bool ok = true;
            if (lane == 0) {
                ok = mbar_wait_inl(&raw_full[i], (uint32_t)(it / raw) & 1u, &abort_flag, err);
                if (ok && it >= stages)
                    ok = mbar_wait_inl(&empty[st], ((uint32_t)(it / stages) & 1u) ^ 1u, &abort_flag, err);
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            const uint8_t *rb = rawbuf + (size_t)i * kQ4RawBytes;
            const __nv_bfloat162 ss =
                q4_scale_pair(reinterpret_cast<const uint16_t *>(rb + kQ4CodeBytes)[row]);
            const __nv_bfloat162 zz = q4_zero_pair(rb[kQ4CodeBytes + 256 + row]);
            const uint4 *codes = reinterpret_cast<const uint4 *>(rb + row * 64);
            uint4 cw[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) cw[q] = codes[(q + rot) & 3];
            uint8_t *wrow = smem + (size_t)st * stage_bytes + row * 128;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int qq = (q + rot) & 3;  // inputs 32 qq .. 32 qq + 31 of the unit
                const uint32_t words[4] = {cw[q].x, cw[q].y, cw[q].z, cw[q].w};
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const int ch = qq * 4 + h;  // inputs 8 ch .. 8 ch + 7
                    *reinterpret_cast<uint4 *>(wrow + (ch >> 3) * kWTileBytes + (((ch & 7) ^ (row & 7)) << 4)) =
                        dequant8_q4(words[h], zz, ss);
                }
            }
            fence_proxy_async_smem();  // the tensor cores read what the threads wrote
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&full[st]);
                mbar_arrive(&raw_empty[i]);
            }
        }
        __syncwarp();
    } else if (warp == 5) {
        // ----------------------------------------------------------------- MMA
        tmem_alloc(tmem_slot, p.tmem_cols);
        tmem_relinquish();
        tc_fence_before_sync();
        named_bar_sync(kBarSetup, kQ4Threads);
        tc_fence_after_sync();
        const uint32_t tmem = *tmem_slot;
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(128, p.ntok);
            int it = 0;
            uint32_t d = tmem;
            for (int u = u0; u < u1; ++u, ++it) {
                const int tile = u / KB, kb = u - tile * KB;
                const int seg = tile - g0;
                const bool seg_first = (kb == 0) || (u == u0);
                if (seg_first) {
                    const int a = seg % n_acc;
                    if (!mbar_wait_inl(&acc_empty[a], ((uint32_t)(seg / n_acc) & 1u) ^ 1u, &abort_flag, err))
                        break;
                    tc_fence_after_sync();
                    d = tmem + (uint32_t)(a * p.ntok);
                }
                const int st = it % stages;
                if (!mbar_wait_inl(&full[st], (uint32_t)(it / stages) & 1u, &abort_flag, err)) break;
                tc_fence_after_sync();
                const uint32_t wa = smem_u32(smem + (size_t)st * stage_bytes);
                const uint32_t xa = wa + w_bytes;
#pragma unroll
                for (int b = 0; b < kBoxes; ++b)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_bf16_ss(d, sdesc_k_sw128(wa + b * kWTileBytes + kk * 32),
                                    sdesc_k_sw128(xa + b * x_box + kk * 32), idesc,
                                    (seg_first && b == 0 && kk == 0) ? 0u : 1u);
                mma_commit(&empty[st]);
                if (u == u1 - 1 || kb == KB - 1) mma_commit(&acc_full[seg % n_acc]);
            }
            mma_commit(drain);
            int dummy = 0;
            mbar_wait(drain, 0, &dummy, err);
        }
        __syncwarp();
    } else {
        // ------------------------------------- warps 0-3: shrink, then epilogue
        decode_epilogue<1>(p, ids, partials, err, c, nseg, acc_full, acc_empty, &abort_flag, red, tmem_slot,
                           kQ4Threads);
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after_sync();
        tmem_dealloc(*tmem_slot, p.tmem_cols);
    }
    trace_exit(trace);
}

// 64 registers: the CTA (352 threads) and two CTAs of the finishing pass fit one SM's
// register file together, so the kernel launched early beside the previous call's
// finishing pass starts on every SM at once (measured: q_proj T = 64 over a 4-bit
// base, 15.8 -> 13.5 us a step with adapters, 12.8 -> 11.4 us base only; at 72
// registers a CTA of the pass no longer fits and the step is back at 15.5 us).
__global__ void __maxnreg__(64)
    gemm_decode_q4_kernel(const __grid_constant__ DecodeMapsQ4 maps, const __grid_constant__ DecodePlanT<1> p,
                          const int32_t *__restrict__ ids, float *__restrict__ partials, int *err)
{
    gemm_decode_q4_body(maps, p, ids, partials, err);
}

// The 4-bit base to bf16, one thread per 8 consecutive inputs of one row (prefill).
__global__ void dequant_q4_kernel(const uint8_t *__restrict__ Wq, const uint16_t *__restrict__ scales,
                                  const uint8_t *__restrict__ zeros, int d_out, int d_in,
                                  uint16_t *__restrict__ W)
{
    const int chunks = d_in / 8;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < (size_t)d_out * chunks;
         i += (size_t)gridDim.x * blockDim.x) {
        const int n = (int)(i / chunks), ch = (int)(i % chunks);
        const int g = ch * 8 / kQ4Group;
        const uint32_t w = *reinterpret_cast<const uint32_t *>(Wq + (size_t)n * (d_in / 2) + ch * 4);
        const uint4 v = dequant8_q4(w, q4_zero_pair(zeros[(size_t)g * d_out + n]),
                                    q4_scale_pair(scales[(size_t)g * d_out + n]));
        *reinterpret_cast<uint4 *>(W + (size_t)n * d_in + ch * 8) = v;
    }
}

constexpr int kFinishThreads = 128;  // each thread: 8 consecutive columns of one token
constexpr int kFinishCols = 8;
constexpr int kFinishBlockCols = kFinishThreads * kFinishCols;
// B pages a finishing thread loads into registers before the GEMM ends (PF): two while
// the finishing grid fits two CTAs per SM beside the GEMM (every CTA is resident and
// loads them early), else one -- fewer registers, four CTAs per SM instead of three
// (measured: T = 256 hot-swap pool 31.7 -> 31.3 us, the grouped 7-module layer 91.1 ->
// 89.3; q_proj T = 64 with one page: 13.5 -> 14.1)
// partial loads in flight per thread, fewer beside the LoRA variant's B words: five
// for one layer (a q_proj tile has ~5.75 contributors; measured 1-3 % faster than four
// on the single-layer workloads), four for a grouped call (five spill there: +1 %)
template <int NP, bool LORA>
constexpr int finish_batch() { return LORA ? (NP == 1 ? 5 : 4) : 8; }

// acc[c] += sum_jj v[jj] * page[n0 + c][jj], the 8 columns' 16-byte words in b[0..7]
__device__ __forceinline__ void expand8(float (&acc)[kFinishCols], const float *v, const uint4 (&b)[8])
{
#pragma unroll
    for (int c = 0; c < kFinishCols; ++c) acc[c] = dot8_f32_bf16(v, b[c], acc[c]);
}

// The pages of adapter slot `id` (0 pages when the slot is not loaded or id is -1).
__device__ __forceinline__ int finish_adapter(const PoolDev &pool, int id, const int32_t *&pages)
{
    if (!slot_loaded(pool.slots, pool.slot_stride, pool.max_adapters, id)) {
        pages = nullptr;
        return 0;
    }
    const int32_t *row = pool.slots + (size_t)id * pool.slot_stride;
    pages = row + SLOT_PAGES;
    return row[SLOT_NPAGES];
}

// The B words of columns n0..n0+7 of the first PF pages into registers, the later
// pages' line into L2.
template <int PF>
__device__ __forceinline__ void finish_b_words(const PoolDev &pool, const int32_t *pages, int np,
                                               int n0, uint4 (&b)[PF][8], int *err)
{
#pragma unroll
    for (int q = 0; q < PF; ++q)
        if (q < np) {
            const int page = LORA_CHECKED(pages[q], 0, pool.num_pages, err, 0);
            const uint16_t *src = pool.B_pages + ((size_t)page * pool.d_out + n0) * kRankPage;
#pragma unroll
            for (int c = 0; c < 8; ++c) b[q][c] = ldg_nc_v4(src + c * kRankPage);
        }
    for (int q = PF; q < np; ++q)
        prefetch_l2(pool.B_pages +
                    ((size_t)LORA_CHECKED(pages[q], 0, pool.num_pages, err, 0) * pool.d_out + n0) *
                        kRankPage);
}

// The sums of one thread's 8 columns of token t (see finish_decode_body).
template <int NP, bool LORA, int PF>
__device__ __forceinline__ void finish_columns(const DecodePlanT<NP> &p, const DecodeProblem &pr,
                                               const float *__restrict__ partials, int t, int n0,
                                               int c_lo, int c_hi, int seg_lo, int np,
                                               const int32_t *pages, bool early,
                                               const uint4 (&b)[PF][8])
{
    const PoolDev &pool = pr.pool;
    const int nl = n0 & 127;

    // One round of loads first: the V values of the pages whose B words are already in
    // registers, the first contributor's partial and the next kFinishBatch ones; the
    // sums and the expand follow in the same order as before (partials in CTA order,
    // then the pages), so the loads of V no longer wait for the partial sums.
    const float *vrow = pr.V + (size_t)t * pr.ldv;
    const int q_early = (LORA && early) ? (np < PF ? np : PF) : 0;
    float4 vq[PF][2];
#pragma unroll
    for (int q = 0; q < PF; ++q)
        if (q < q_early) {
            vq[q][0] = *reinterpret_cast<const float4 *>(vrow + q * kRankPage);
            vq[q][1] = *reinterpret_cast<const float4 *>(vrow + q * kRankPage + 4);
        }
    float acc[kFinishCols];
    {
        const float *src = partials + (((size_t)c_lo * p.max_seg + seg_lo) * p.T + t) * 128 + nl;
        const float4 a0 = *reinterpret_cast<const float4 *>(src);
        const float4 a1 = *reinterpret_cast<const float4 *>(src + 4);
        acc[0] = a0.x; acc[1] = a0.y; acc[2] = a0.z; acc[3] = a0.w;
        acc[4] = a1.x; acc[5] = a1.y; acc[6] = a1.z; acc[7] = a1.w;
    }
    // the other contributors' first partials, kFinishBatch loads in flight at a time
    // (summed in CTA order all the same)
    const size_t stride = (size_t)p.max_seg * p.T * 128;
    const float *src = partials + ((size_t)(c_lo + 1) * p.max_seg * p.T + t) * 128 + nl;
    constexpr int kFinishBatch = finish_batch<NP, LORA>();
    for (int c0 = c_lo + 1; c0 <= c_hi; c0 += kFinishBatch, src += kFinishBatch * stride) {
        float4 v[kFinishBatch][2];
#pragma unroll
        for (int i = 0; i < kFinishBatch; ++i)
            if (c0 + i <= c_hi) {
                v[i][0] = *reinterpret_cast<const float4 *>(src + i * stride);
                v[i][1] = *reinterpret_cast<const float4 *>(src + i * stride + 4);
            }
#pragma unroll
        for (int i = 0; i < kFinishBatch; ++i)
            if (c0 + i <= c_hi) {
                acc[0] += v[i][0].x; acc[1] += v[i][0].y; acc[2] += v[i][0].z; acc[3] += v[i][0].w;
                acc[4] += v[i][1].x; acc[5] += v[i][1].y; acc[6] += v[i][1].z; acc[7] += v[i][1].w;
            }
    }
#pragma unroll
    for (int q = 0; q < PF; ++q)
        if (q < q_early) {
            const float v[8] = {vq[q][0].x, vq[q][0].y, vq[q][0].z, vq[q][0].w,
                                vq[q][1].x, vq[q][1].y, vq[q][1].z, vq[q][1].w};
            expand8(acc, v, b[q]);
        }
    for (int q = q_early; q < np; ++q) {
        float v[8];
        const float4 v0 = *reinterpret_cast<const float4 *>(vrow + q * kRankPage);
        const float4 v1 = *reinterpret_cast<const float4 *>(vrow + q * kRankPage + 4);
        v[0] = v0.x; v[1] = v0.y; v[2] = v0.z; v[3] = v0.w;
        v[4] = v1.x; v[5] = v1.y; v[6] = v1.z; v[7] = v1.w;
        {
            uint4 bq[8];
            const int page = LORA_CHECKED(pages[q], 0, pool.num_pages, pr.err, 0);
            const uint16_t *bsrc = pool.B_pages + ((size_t)page * pool.d_out + n0) * kRankPage;
#pragma unroll
            for (int c = 0; c < 8; ++c) bq[c] = ldg_nc_v4(bsrc + c * kRankPage);
            expand8(acc, v, bq);
        }
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]);
    o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]);
    o.w = pack_bf16x2(acc[6], acc[7]);
    *reinterpret_cast<uint4 *>(pr.Y + (size_t)t * pool.d_out + n0) = o;
}

// LORA = false: the base-only pass (no adapter state, few registers).
template <int NP, bool LORA, int PF>
__device__ __forceinline__ void finish_decode_body(const DecodePlanT<NP> &p,
                                                   const float *__restrict__ partials,
                                                   const int32_t *__restrict__ ids)
{
    // The next call's GEMM may launch now: its CTAs take an SM as soon as this call's
    // GEMM CTA leaves it and stream their first W tiles; everything they write comes
    // after their own wait for this kernel.
    pdl_launch_dependents();
    uint64_t *const trace = p.trace ? p.trace + 3 * kTraceWords : nullptr;  // kernel slot 3
    trace_enter(trace);
    int m = 0;
    for (int k = 1; NP > 1 && k < p.n; ++k)
        if (p.prob[pick<NP>(k)].col_blk_begin <= (int)blockIdx.x) m = k;
    const DecodeProblem &pr = p.prob[pick<NP>(m)];
    const PoolDev &pool = pr.pool;
    const int n0 = ((blockIdx.x - pr.col_blk_begin) * kFinishThreads + threadIdx.x) * kFinishCols;
    const int t = blockIdx.y;
    const bool col_ok = n0 < pool.d_out;  // d_out is a multiple of 8

    // ---- ahead of the GEMM kernel's end: this token's adapter and its B words (the
    // 8 columns' 16-byte words of a page are one 128-byte line): the first pages into
    // registers, the rest into L2. The id read here may still be written by a kernel
    // ahead of the GEMM in the stream, so it is read again after the wait and the
    // words are reloaded if it changed.
    int id = -1, np = 0;
    const int32_t *pages = nullptr;
    uint4 b[PF][8];
    if (LORA && pool.slots != nullptr) {
        id = ids[t];
        np = finish_adapter(pool, id, pages);
        if (col_ok) finish_b_words<PF>(pool, pages, np, n0, b, pr.err);
    }
    // contributors of this tile: CTAs c_lo..c_hi (contiguous unit ranges). Only c_lo
    // can have started before the tile; its partial for the tile is its segment
    // (tile - its first tile), the others' is their segment 0. (U * G < 2^31 is
    // checked on the host, so the products fit in 32 bits.)
    const int tile = n0 >> 7;
    const int ub = pr.u_begin + tile * pr.KB, ue = ub + pr.KB;
    int c_lo = (ub * p.G) / p.U;
    while (c_lo > 0 && (c_lo * p.U) / p.G > ub) --c_lo;
    while (((c_lo + 1) * p.U) / p.G <= ub) ++c_lo;
    int c_hi = c_lo;
    while (c_hi + 1 < p.G && ((c_hi + 1) * p.U) / p.G < ue) ++c_hi;
    int seg_lo = pr.g_begin + tile - unit_tile(p, (c_lo * p.U) / p.G);
#ifdef LORA_CHECK
    // the split-K slots this thread reads: contributors within the ranges, the first
    // one's segment within its partials
    if (col_ok && (!check_range(c_lo, 0, p.G, pr.err) || !check_range(c_hi, c_lo, p.G, pr.err) ||
                   !check_range(seg_lo, 0, p.max_seg, pr.err))) {
        c_lo = c_hi = 0;
        seg_lo = 0;
    }
#endif

    // ---- partials and V are written by the GEMM kernel
    pdl_wait_prior();
    if (threadIdx.x == 0) trace_release(trace);
    bool early = true;  // the words in b belong to this token's adapter
    if (LORA && pool.slots != nullptr) {
        const int id_now = ids[t];
        if (id_now != id) {
            id = id_now;
            np = finish_adapter(pool, id, pages);
            early = false;
        }
        if (np == 0 && id != -1 && threadIdx.x == 0 && (int)blockIdx.x == pr.col_blk_begin)
            atomicOr(pr.err, kErrBadIdBit);  // strict: never a silent base fall-back
    }
    if (col_ok) finish_columns<NP, LORA, PF>(p, pr, partials, t, n0, c_lo, c_hi, seg_lo, np, pages, early, b);
    if (trace) {
        __syncthreads();
        trace_exit(trace);
    }
}

// Register budgets. The register file is split among an SM's four sub-partitions
// (16384 registers each) and a CTA's warps are dealt to them in turn, so the six
// GEMM warps put two warps on two sub-partitions. When the adapter finishing pass
// has more CTAs than there are SMs, two of its CTAs (one warp per sub-partition
// each) must fit beside a GEMM CTA to be resident, with their B words loaded,
// when the GEMM ends: 2 x 96 x 32 + 2 x 152 x 32 <= 16384. Measured on q_proj
// (T = 64, 256 finishing CTAs): without the bounds only 152 were resident, the
// other 104 and then a quarter of the next call's GEMM CTAs started only as GEMM
// CTAs left (15.7 vs 17.2 us a step). The bounds cost registers the shrink and the
// partial loads use, so they are taken only where they pay: the finishing grid
// exceeds the SMs and a CTA's shrink pairs read at most half as many bytes as its
// share of W (the "tight" plans; measured faster for q_proj T = 64, gate_proj
// T = 32 and the grouped 7-module layer; slower for T = 32 layers whose finishing
// grid fits the SMs and for T = 256 with ~4 shrink pairs per CTA). The unbounded
// finishing pass is still held to three CTAs per SM (168 registers): at 180 its
// residency fell to two and T = 256 took 38 instead of 34.6 us a step. The unbounded
// GEMM keeps four chunks of shrink loads in flight per thread (146 registers, two
// unbounded finishing CTAs still fit beside it): T = 256 over 2000 adapters, where
// the shrink of ~3.4 pairs per CTA outlasts the MMAs, 28.6 -> 27.7 us a step (three
// chunks: 28.5); the tight variant keeps two.
template <int NP>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_decode_kernel(const __grid_constant__ DecodeMapsT<NP> maps,
                       const __grid_constant__ DecodePlanT<NP> p, const int32_t *__restrict__ ids,
                       float *__restrict__ partials, int *err)
{
    gemm_decode_body<NP, 4>(maps, p, ids, partials, err);
}

template <int NP>
__global__ void __maxnreg__(96)
    gemm_decode_kernel_tight(const __grid_constant__ DecodeMapsT<NP> maps,
                             const __grid_constant__ DecodePlanT<NP> p,
                             const int32_t *__restrict__ ids, float *__restrict__ partials, int *err)
{
    gemm_decode_body<NP>(maps, p, ids, partials, err);
}

template <int NP, bool LORA, int PF>
__global__ void __launch_bounds__(kFinishThreads, 3)
    finish_decode_kernel(const __grid_constant__ DecodePlanT<NP> p, const float *__restrict__ partials,
                         const int32_t *__restrict__ ids)
{
    finish_decode_body<NP, LORA, PF>(p, partials, ids);
}

template <int NP, int PF>
__global__ void __maxnreg__(152)
    finish_decode_kernel_tight(const __grid_constant__ DecodePlanT<NP> p,
                               const float *__restrict__ partials, const int32_t *__restrict__ ids)
{
    finish_decode_body<NP, true, PF>(p, partials, ids);
}

uint32_t pow2_cols(uint32_t n)
{
    uint32_t c = 32;
    while (c < n) c <<= 1;
    return c;
}

// programmatic stream serialization: the kernel's prologue (and, for the GEMM,
// its first W tiles) overlaps the previous kernel in the stream; each kernel
// waits (griddepcontrol.wait) before it touches anything the stream wrote
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace

bool plan_decode(int n, int T, const int *d_in, const int *d_out, const int *max_pages, int max_G,
                 DecodePlan *out)
{
    if (n < 1 || n > kMaxGroup || T < 1 || T > kDecodeMaxT || max_G < 1) return false;
    DecodePlan p{};
    p.n = n;
    p.T = T;
    p.ntok = ((T + 15) / 16) * 16;
    long long U = 0, pairs = 0, cols = 0;
    int g = 0;
    for (int m = 0; m < n; ++m) {
        DecodeProblem &q = p.prob[m];
        q.KB = (d_in[m] + 64 * kBoxes - 1) / (64 * kBoxes);
        q.n_tiles = (d_out[m] + 127) / 128;
        q.u_begin = (int)U;
        q.g_begin = g;
        q.pair_begin = (int)pairs;
        q.col_blk_begin = (int)cols;
        U += (long long)q.n_tiles * q.KB;
        g += q.n_tiles;
        pairs += (long long)T * max_pages[m];
        cols += (d_out[m] + kFinishBlockCols - 1) / kFinishBlockCols;
    }
    long long G = max_G < U ? max_G : U;
    // the finishing pass computes c * U in 32 bits
    if (U * G >= (1ll << 31) || pairs >= (1ll << 31) || cols >= (1ll << 31)) return false;
    p.U = (int)U;
    p.G = (int)G;
    // more CTAs than ranges when the shrink pairs outnumber them (small layers)
    p.grid = p.G;
    if (pairs > p.grid) p.grid = (int)(pairs < max_G ? pairs : max_G);
    p.pairs = (int)pairs;
    p.col_blocks = (int)cols;
    p.fin_two_pages = cols * T <= 2ll * max_G;
    // bounded registers where the finishing grid exceeds the SMs and each CTA's
    // shrink work (A bytes of its pairs) stays well under its share of the W stream
    int max_d_in = 0;
    for (int m = 0; m < n; ++m) max_d_in = d_in[m] > max_d_in ? d_in[m] : max_d_in;
    const double shrink_bytes = (double)((pairs + p.grid - 1) / p.grid) * 2.0 * kRankPage * max_d_in;
    const double stream_bytes = (double)U / (double)G * kBoxes * kWTileBytes;
    p.tight = pairs > 0 && cols * T > max_G && 2.0 * shrink_bytes <= stream_bytes;
    // the A pages requested into L2 before the wait on the previous kernel, one bulk
    // prefetch per page: faster for every plan measured (T = 256 over 2000 adapters,
    // ~3.4 pairs per CTA: 31.3 -> 28.7 us a step; q_proj T = 64: 13.49 -> 13.35; the
    // 7-module layer 89.3 -> 89.0). Line prefetches by the epilogue warps had paid only
    // where a CTA's pairs were few (T = 256: 34 -> 37 us with them)
    p.prefetch_a = pairs > 0;
    int max_seg = 1;
    for (int c = 0; c < p.G; ++c) {
        const int u0 = cta_start(c, p.U, p.G), u1 = cta_start(c + 1, p.U, p.G);
        const int s = unit_tile(p, u1 - 1) - unit_tile(p, u0) + 1;
        if (s > max_seg) max_seg = s;
    }
    p.max_seg = max_seg;
    // accumulators: one per segment of a range, within the 512 TMEM columns
    int n_acc = 512 / p.ntok;
    if (n_acc > max_seg) n_acc = max_seg;
    p.n_acc = n_acc;
    const size_t stage_bytes = kBoxes * (kWTileBytes + (size_t)p.ntok * 128);
    int stages = (int)((200 * 1024) / stage_bytes);
    if (stages > 8) stages = 8;
    if (stages < 2) stages = 2;
    p.stages = stages;
    p.smem_bytes = 1024 + stages * stage_bytes + (2 * stages + 2 * n_acc + 1) * 8 + 16;
    p.tmem_cols = pow2_cols((uint32_t)(n_acc * p.ntok));
    *out = p;
    return true;
}

size_t decode_partials_floats(const DecodePlan &p) { return (size_t)p.G * p.max_seg * p.T * 128; }

namespace {

template <int NP>
DecodePlanT<NP> narrow_plan(const DecodePlan &p)
{
    DecodePlanT<NP> q{};
    static_cast<DecodePlanHead &>(q) = static_cast<const DecodePlanHead &>(p);
    for (int m = 0; m < NP; ++m) q.prob[m] = p.prob[m];
    return q;
}

template <int NP>
cudaError_t launch_gemm_decode_n(const DecodeMaps &maps, const DecodePlan &plan, const int32_t *ids,
                                 float *partials, int *err, cudaStream_t stream)
{
    auto kernel = plan.tight ? gemm_decode_kernel_tight<NP> : gemm_decode_kernel<NP>;
    cudaError_t e = ensure_smem_attr((const void *)kernel, plan.smem_bytes);
    if (e != cudaSuccess) return e;
    DecodeMapsT<NP> m;
    for (int i = 0; i < NP; ++i) {
        m.W[i] = maps.W[i];
        m.X[i] = maps.X[i];
    }
    return launch_pdl(kernel, dim3(plan.grid), dim3(kThreads), plan.smem_bytes, stream, m,
                      narrow_plan<NP>(plan), ids, partials, err);
}

template <int NP>
cudaError_t launch_finish_decode_n(const DecodePlan &plan, const float *partials, const int32_t *ids,
                                   cudaStream_t stream)
{
    auto kernel = ids == nullptr   ? finish_decode_kernel<NP, false, 1>
                  : plan.fin_two_pages ? (plan.tight ? finish_decode_kernel_tight<NP, 2> : finish_decode_kernel<NP, true, 2>)
                                       : (plan.tight ? finish_decode_kernel_tight<NP, 1> : finish_decode_kernel<NP, true, 1>);
    cudaError_t e = ensure_smem_attr((const void *)kernel, 0);
    if (e != cudaSuccess) return e;
    return launch_pdl(kernel, dim3(plan.col_blocks, plan.T), dim3(kFinishThreads), 0, stream,
                      narrow_plan<NP>(plan), partials, ids);
}

}  // namespace

cudaError_t launch_gemm_decode(const DecodeMaps &maps, const DecodePlan &plan, const int32_t *ids,
                               float *partials, int *err, cudaStream_t stream)
{
    if (plan.n == 1) return launch_gemm_decode_n<1>(maps, plan, ids, partials, err, stream);
    return launch_gemm_decode_n<kMaxGroup>(maps, plan, ids, partials, err, stream);
}

cudaError_t launch_finish_decode(const DecodePlan &plan, const float *partials, const int32_t *ids,
                                 cudaStream_t stream)
{
    if (plan.n == 1) return launch_finish_decode_n<1>(plan, partials, ids, stream);
    return launch_finish_decode_n<kMaxGroup>(plan, partials, ids, stream);
}

bool plan_decode_q4(DecodePlan *plan)
{
    DecodePlan &p = *plan;
    if (p.n != 1 || p.prob[0].KB * 128 != p.prob[0].pool.d_in) return false;
    constexpr size_t kMaxSmem = 232448;  // per CTA on this GPU
    const size_t stage_bytes = kBoxes * (kWTileBytes + (size_t)p.ntok * 128);
    for (int stages = 3; stages >= 2; --stages) {
        const size_t fixed = 1024 + stages * stage_bytes + 512;
        if (fixed + 2 * kQ4RawBytes > kMaxSmem) continue;
        int raw = (int)((kMaxSmem - fixed) / kQ4RawBytes);
        if (raw > 5) raw = 5;  // five units of codes in flight (measured no slower than eight)
        p.stages = stages;
        p.raw_stages = raw;
        p.smem_bytes = 1024 + stages * stage_bytes + (size_t)raw * kQ4RawBytes +
                       (2 * stages + 2 * raw + 2 * p.n_acc + 1) * 8 + 16;
        return p.smem_bytes <= kMaxSmem;
    }
    return false;
}

cudaError_t launch_gemm_decode_q4(const DecodeMapsQ4 &maps, const DecodePlan &plan, const int32_t *ids,
                                  float *partials, int *err, cudaStream_t stream)
{
    cudaError_t e = ensure_smem_attr((const void *)gemm_decode_q4_kernel, plan.smem_bytes);
    if (e != cudaSuccess) return e;
    return launch_pdl(gemm_decode_q4_kernel, dim3(plan.grid), dim3(kQ4Threads), plan.smem_bytes, stream, maps,
                      narrow_plan<1>(plan), ids, partials, err);
}

cudaError_t launch_dequant_q4(const uint8_t *Wq, const uint16_t *scales, const uint8_t *zeros, int d_out,
                              int d_in, uint16_t *W, cudaStream_t stream)
{
    cudaError_t e = ensure_smem_attr((const void *)dequant_q4_kernel, 0);
    if (e != cudaSuccess) return e;
    const size_t chunks = (size_t)d_out * (d_in / 8);
    const int grid = (int)std::min<size_t>((chunks + 255) / 256, 152 * 16);
    dequant_q4_kernel<<<grid, 256, 0, stream>>>(Wq, scales, zeros, d_out, d_in, W);
    return cudaGetLastError();
}

}  // namespace lora
