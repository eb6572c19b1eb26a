// gemm_decode.cu -- the decode path (T <= 256): two kernels.
//
// 1. gemm_decode_kernel: base product + the per-token low-rank shrink.
//    At decode sizes the base GEMM is bound by reading W_base once from HBM, so
//    the layout is chosen to stream W at full bandwidth on every SM:
//    * operands swapped: D[n, t] = sum_k W[n,k] X[t,k], so the long d_out side
//      is the MMA's M (128 rows of W per tile) and the T tokens are its N
//      (T rounded up to 16; rows past T read as zero from TMA);
//    * stream-K: the (tile, 128-wide k-block) iteration space is cut into G
//      equal contiguous ranges, one per CTA (G = number of SMs, or fewer for
//      small problems), so every SM streams the same share of W. A range
//      touches at most two tiles; each touched tile gets its own TMEM
//      accumulator and is written as an fp32 partial sum [cta][0|1][T][128];
//    * warp roles: warp 4 issues TMA loads (per stage two W boxes 128x64 and two
//      X boxes T'x64, 128-byte swizzle) into a multi-stage ring and starts before TMEM is
//      allocated; warp 5 allocates TMEM and issues tcgen05 MMAs (M=128, N=T',
//      K=16); warps 0-3, idle until the accumulators are ready, first compute
//      the low-rank shrink V[t, 8q..8q+7] = s_i X[t,:] A_i[:, 8q..8q+7] for
//      the (token, page) pairs dealt to this CTA round-robin (a BGMV-style
//      per-token gather: each pair reads one 8 x d_in A page with 128-bit
//      loads), so the adapter reads overlap the W stream; then they read the
//      accumulators back with tcgen05.ld (TMEM lane = output row n) and store
//      the partials.
// 2. finish_decode_kernel (launched with programmatic stream serialization, so
//    it is resident and has prefetched its B pages before the GEMM ends): per
//    output element, the partials of the CTAs that covered its tile are summed
//    in CTA order (deterministic), the low-rank expand s_i V[t,:] B_i[:,n] is
//    added from the interleaved B pages (one 16-byte load = 8 rank rows of one
//    column; V already carries s_i), and the sum is rounded once to bf16.
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

struct ShrinkArgs {
    const uint16_t *X;
    const int32_t *ids;  // nullptr: base product only
    float *V;
    int ldv;
};

// One (token, page) pair of the shrink, computed by the 128 threads of warps 0-3.
__device__ __forceinline__ void shrink_pair(int t, int page, float scale, const PoolDev &pool,
                                            const ShrinkArgs &sa, int q, float (*red)[8])
{
    const int tid = threadIdx.x;  // 0..127
    const int warp = tid >> 5, lane = tid & 31;
    const int d_in = pool.d_in;
    const uint16_t *Ap = pool.A_pages + (size_t)page * kRankPage * d_in;
    const uint16_t *xr = sa.X + (size_t)t * d_in;
    float acc[kRankPage];
#pragma unroll
    for (int jj = 0; jj < kRankPage; ++jj) acc[jj] = 0.f;
#pragma unroll 2
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
        sa.V[(size_t)t * sa.ldv + q * kRankPage + tid] = scale * s;
    }
    named_bar_sync(kBarShrink, 128);
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_decode_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                       DecodePlan p, float *__restrict__ partials, int *err, PoolDev pool,
                       ShrinkArgs sa)
{
    extern __shared__ uint8_t dec_smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(dec_smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t x_box = (uint32_t)p.ntok * 128;  // one TMA box of X
    const uint32_t w_bytes = kBoxes * kWTileBytes;
    const uint32_t stage_bytes = w_bytes + kBoxes * x_box;
    const int stages = p.stages;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)stages * stage_bytes);
    uint64_t *empty = full + stages;
    uint64_t *acc_full = empty + stages;  // [2]
    uint64_t *drain = acc_full + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    __shared__ int abort_flag;
    __shared__ float red[4][kRankPage];

    // the finishing kernel may start its independent prologue now
    pdl_launch_dependents();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.x;
    const int u0 = cta_start(c, p.U, p.G), u1 = cta_start(c + 1, p.U, p.G);
    const int tile0 = u0 / p.KB;
    const int nseg = (u1 > u0) ? (u1 - 1) / p.KB - tile0 + 1 : 0;

    if (warp == 4) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            for (int i = 0; i < stages; ++i) {
                mbar_init(&full[i], 1);
                mbar_init(&empty[i], 1);
            }
            mbar_init(&acc_full[0], 1);
            mbar_init(&acc_full[1], 1);
            mbar_init(drain, 1);
            abort_flag = 0;
            fence_mbar_init();
            tma_prefetch_map(&tmW);
            tma_prefetch_map(&tmX);
        }
        __syncwarp();
        named_bar_arrive(kBarSetup, kThreads);  // barriers are ready; do not wait for TMEM
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();  // W is read exactly once
            // W is a weight: the first ring's worth of W tiles is requested before the
            // previous kernel in the stream has finished; X (and everything the epilogue
            // touches) only after the programmatic wait.
            const int pre = (u1 - u0) < stages ? (u1 - u0) : stages;
            for (int i = 0; i < pre; ++i) {
                const int u = u0 + i, tile = u / p.KB, kb = u - tile * p.KB;
                mbar_arrive_expect_tx(&full[i], stage_bytes);
                for (int b = 0; b < kBoxes; ++b)
                    tma_load_2d_hint(smem + (size_t)i * stage_bytes + b * kWTileBytes, &tmW, &full[i],
                                     (kb * kBoxes + b) * 64, tile * 128, pol_w);
            }
            pdl_wait_prior();
            for (int i = 0; i < pre; ++i) {
                const int kb = (u0 + i) % p.KB;
                for (int b = 0; b < kBoxes; ++b)
                    tma_load_2d(smem + (size_t)i * stage_bytes + w_bytes + b * x_box, &tmX, &full[i],
                                (kb * kBoxes + b) * 64, 0);
            }
            int it = pre;
            for (int u = u0 + pre; u < u1; ++u, ++it) {
                const int s = it % stages;
                if (!mbar_wait(&empty[s], ((uint32_t)(it / stages) & 1u) ^ 1u, &abort_flag, err)) break;
                const int tile = u / p.KB, kb = u - tile * p.KB;
                uint8_t *ws = smem + (size_t)s * stage_bytes;
                mbar_arrive_expect_tx(&full[s], stage_bytes);
                for (int b = 0; b < kBoxes; ++b) {
                    tma_load_2d_hint(ws + b * kWTileBytes, &tmW, &full[s], (kb * kBoxes + b) * 64,
                                     tile * 128, pol_w);
                    tma_load_2d(ws + w_bytes + b * x_box, &tmX, &full[s], (kb * kBoxes + b) * 64, 0);
                }
            }
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
            for (int u = u0; u < u1; ++u, ++it) {
                const int s = it % stages;
                if (!mbar_wait(&full[s], (uint32_t)(it / stages) & 1u, &abort_flag, err)) break;
                tc_fence_after_sync();
                const int tile = u / p.KB, kb = u - tile * p.KB;
                const int seg = tile - tile0;
                const uint32_t d = tmem + (uint32_t)(seg * p.ntok);
                const uint32_t wa = smem_u32(smem + (size_t)s * stage_bytes);
                const uint32_t xa = wa + w_bytes;
                const bool first = (kb == 0) || (u == u0);
#pragma unroll
                for (int b = 0; b < kBoxes; ++b)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_bf16_ss(d, sdesc_k_sw128(wa + b * kWTileBytes + kk * 32),
                                    sdesc_k_sw128(xa + b * x_box + kk * 32), idesc,
                                    (first && b == 0 && kk == 0) ? 0u : 1u);
                mma_commit(&empty[s]);
                if (u == u1 - 1 || kb == p.KB - 1) mma_commit(&acc_full[seg]);
            }
            mma_commit(drain);
            int dummy = 0;
            mbar_wait(drain, 0, &dummy, err);
        }
        __syncwarp();
    } else {
        // ------------------------------------- warps 0-3: shrink, then epilogue
        named_bar_sync(kBarSetup, kThreads);
        tc_fence_after_sync();
        const uint32_t tmem = *tmem_slot;
        pdl_wait_prior();  // X, ids, V and the partials belong to the stream's order
        if (sa.ids != nullptr) {
            const int pairs = p.T * pool.max_pages;
            for (int u = c; u < pairs; u += p.G) {
                const int t = u / pool.max_pages, q = u - t * pool.max_pages;
                const int id = sa.ids[t];
                if (!slot_loaded(pool.slots, pool.slot_stride, pool.max_adapters, id)) continue;
                const int32_t *row = pool.slots + (size_t)id * pool.slot_stride;
                if (q >= row[SLOT_NPAGES]) continue;
                shrink_pair(t, row[SLOT_PAGES + q], __int_as_float(row[SLOT_SCALE]), pool, sa, q,
                            red);
            }
        }
        for (int seg = 0; seg < nseg; ++seg) {
            bool ok = true;
            if (lane == 0) ok = mbar_wait(&acc_full[seg], 0, &abort_flag, err);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after_sync();
            float *out = partials + (size_t)(c * 2 + seg) * p.T * 128 + warp * 32 + lane;
            for (int col = 0; col < p.ntok; col += 16) {
                uint32_t v[16];
                tmem_ld16_wait(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(seg * p.ntok + col), v);
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (col + j < p.T) out[(size_t)(col + j) * 128] = __uint_as_float(v[j]);
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after_sync();
        tmem_dealloc(*tmem_slot, p.tmem_cols);
    }
}

constexpr int kFinishThreads = 128;  // each thread: 8 consecutive columns of one token
constexpr int kFinishCols = 8;
constexpr int kPrefetchPages = 2;     // B pages fetched before the GEMM has finished
constexpr int kFinishBatch = 8;       // partial loads in flight per thread

__device__ __forceinline__ void add8(float (&acc)[kFinishCols], const float *src)
{
    const float4 a = *reinterpret_cast<const float4 *>(src);
    const float4 b = *reinterpret_cast<const float4 *>(src + 4);
    acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
    acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
}

// acc[c] += sum_jj v[jj] * page[n0 + c][jj], the 8 columns' 16-byte words in b[0..7]
__device__ __forceinline__ void expand8(float (&acc)[kFinishCols], const float *v, const uint4 (&b)[8])
{
#pragma unroll
    for (int c = 0; c < kFinishCols; ++c) acc[c] = dot8_f32_bf16(v, b[c], acc[c]);
}

__global__ void __launch_bounds__(kFinishThreads)
    finish_decode_kernel(DecodePlan p, const float *__restrict__ partials,
                         const int32_t *__restrict__ ids, PoolDev pool, const float *__restrict__ V,
                         int ldv, uint16_t *__restrict__ Y, int *err)
{
    // The next call's GEMM may launch now: its CTAs take an SM as soon as this call's
    // GEMM CTA leaves it and stream their first W tiles; everything they write comes
    // after their own wait for this kernel.
    pdl_launch_dependents();
    const int n0 = (blockIdx.x * kFinishThreads + threadIdx.x) * kFinishCols;
    const int t = blockIdx.y;
    const bool col_ok = n0 < pool.d_out;  // d_out is a multiple of 8

    // ---- independent of the GEMM kernel: this token's adapter and its first B words
    int np = 0;
    const int32_t *pages = nullptr;
    if (ids != nullptr) {
        const int id = ids[t];
        if (slot_loaded(pool.slots, pool.slot_stride, pool.max_adapters, id)) {
            const int32_t *row = pool.slots + (size_t)id * pool.slot_stride;
            np = row[SLOT_NPAGES];
            pages = row + SLOT_PAGES;
        } else if (id != -1 && threadIdx.x == 0 && blockIdx.x == 0) {
            atomicOr(err, kErrBadIdBit);  // strict: never a silent base fall-back
        }
    }
    uint4 b[kPrefetchPages][8];
    if (col_ok) {
#pragma unroll
        for (int q = 0; q < kPrefetchPages; ++q)
            if (q < np) {
                const uint16_t *src = pool.B_pages + ((size_t)pages[q] * pool.d_out + n0) * kRankPage;
#pragma unroll
                for (int c = 0; c < 8; ++c) b[q][c] = ldg_nc_v4(src + c * kRankPage);
            }
    }
    // contributors of this tile: CTAs c_lo..c_hi (contiguous k-ranges); only c_lo can
    // have started in the previous tile, in which case its partial for this tile is
    // its second one. (U < 2^20 and G < 2^11, so the products fit in 32 bits.)
    const int tile = n0 >> 7, nl = n0 & 127;
    const int kb_lo = tile * p.KB, kb_hi = kb_lo + p.KB;
    int c_lo = (kb_lo * p.G) / p.U;
    while (c_lo > 0 && (c_lo * p.U) / p.G > kb_lo) --c_lo;
    while (((c_lo + 1) * p.U) / p.G <= kb_lo) ++c_lo;
    int c_hi = c_lo;
    while (c_hi + 1 < p.G && ((c_hi + 1) * p.U) / p.G < kb_hi) ++c_hi;
    const int seg_lo = (c_lo * p.U) / p.G < kb_lo ? 1 : 0;

    // ---- partials and V are written by the GEMM kernel
    pdl_wait_prior();
    if (!col_ok) return;

    float acc[kFinishCols] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    add8(acc, partials + ((size_t)(c_lo * 2 + seg_lo) * p.T + t) * 128 + nl);
    // the other contributors' first partials, kFinishBatch loads in flight at a time
    // (summed in CTA order all the same)
    const size_t stride = (size_t)2 * p.T * 128;
    const float *src = partials + ((size_t)(c_lo + 1) * 2 * p.T + t) * 128 + nl;
    for (int c0 = c_lo + 1; c0 <= c_hi; c0 += kFinishBatch, src += kFinishBatch * stride) {
        float4 b[kFinishBatch][2];
#pragma unroll
        for (int i = 0; i < kFinishBatch; ++i)
            if (c0 + i <= c_hi) {
                b[i][0] = *reinterpret_cast<const float4 *>(src + i * stride);
                b[i][1] = *reinterpret_cast<const float4 *>(src + i * stride + 4);
            }
#pragma unroll
        for (int i = 0; i < kFinishBatch; ++i)
            if (c0 + i <= c_hi) {
                acc[0] += b[i][0].x; acc[1] += b[i][0].y; acc[2] += b[i][0].z; acc[3] += b[i][0].w;
                acc[4] += b[i][1].x; acc[5] += b[i][1].y; acc[6] += b[i][1].z; acc[7] += b[i][1].w;
            }
    }
    const float *vrow = V + (size_t)t * ldv;
    for (int q = 0; q < np; ++q) {
        float v[8];
        const float4 v0 = *reinterpret_cast<const float4 *>(vrow + q * kRankPage);
        const float4 v1 = *reinterpret_cast<const float4 *>(vrow + q * kRankPage + 4);
        v[0] = v0.x; v[1] = v0.y; v[2] = v0.z; v[3] = v0.w;
        v[4] = v1.x; v[5] = v1.y; v[6] = v1.z; v[7] = v1.w;
        if (q < kPrefetchPages) {
            if (q == 0) expand8(acc, v, b[0]);
            else expand8(acc, v, b[1]);
        } else {
            uint4 bq[8];
            const uint16_t *src = pool.B_pages + ((size_t)pages[q] * pool.d_out + n0) * kRankPage;
#pragma unroll
            for (int c = 0; c < 8; ++c) bq[c] = ldg_nc_v4(src + c * kRankPage);
            expand8(acc, v, bq);
        }
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]);
    o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]);
    o.w = pack_bf16x2(acc[6], acc[7]);
    *reinterpret_cast<uint4 *>(Y + (size_t)t * pool.d_out + n0) = o;
}

uint32_t pow2_cols(uint32_t n)
{
    uint32_t c = 32;
    while (c < n) c <<= 1;
    return c;
}

}  // namespace

DecodePlan plan_decode(int T, int d_in, int d_out, int num_sms)
{
    DecodePlan p{};
    p.T = T;
    p.ntok = ((T + 15) / 16) * 16;
    if (p.ntok < 16) p.ntok = 16;
    p.KB = (d_in + 64 * kBoxes - 1) / (64 * kBoxes);
    p.n_tiles = (d_out + 127) / 128;
    p.U = p.n_tiles * p.KB;
    int G = num_sms;
    if (G > p.U) G = p.U;
    if (G < p.n_tiles) G = p.n_tiles;  // ranges never span more than two tiles
    p.G = G;
    const size_t stage_bytes = kBoxes * (kWTileBytes + (size_t)p.ntok * 128);
    int stages = (int)((200 * 1024) / stage_bytes);
    if (stages > 8) stages = 8;
    if (stages < 2) stages = 2;
    p.stages = stages;
    p.smem_bytes = 1024 + stages * stage_bytes + (2 * stages + 3) * 8 + 16;
    p.tmem_cols = pow2_cols(2 * p.ntok);
    return p;
}

size_t decode_partials_floats(const DecodePlan &p) { return (size_t)p.G * 2 * p.T * 128; }

cudaError_t launch_gemm_decode(const CUtensorMap &tmW, const CUtensorMap &tmX,
                               const DecodePlan &plan, const PoolDev &pool, const uint16_t *X,
                               const int32_t *ids, float *V, int ldv, float *partials, int *err,
                               cudaStream_t stream)
{
    cudaError_t e = ensure_smem_attr((const void *)gemm_decode_kernel, plan.smem_bytes);
    if (e != cudaSuccess) return e;
    ShrinkArgs sa{X, ids, V, ldv};
    // programmatic stream serialization: the prologue and the first W tiles overlap the
    // previous kernel in the stream (the kernel waits before touching anything else)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.G);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = plan.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemm_decode_kernel, tmW, tmX, plan, partials, err, pool, sa);
}

cudaError_t launch_finish_decode(const DecodePlan &plan, const float *partials,
                                 const int32_t *ids, const PoolDev &pool, const float *V,
                                 int ldv, uint16_t *Y, int *err, cudaStream_t stream)
{
    cudaError_t e = ensure_smem_attr((const void *)finish_decode_kernel, 0);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    const int per_cta = kFinishThreads * kFinishCols;
    cfg.gridDim = dim3((pool.d_out + per_cta - 1) / per_cta, plan.T);
    cfg.blockDim = dim3(kFinishThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, finish_decode_kernel, plan, partials, ids, pool, V, ldv, Y, err);
}

}  // namespace lora
