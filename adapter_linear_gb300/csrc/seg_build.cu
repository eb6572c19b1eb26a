// seg_build.cu -- segment builder: the "Grouped Multi-LoRA Execution" step of
// the LoRA-Land blog (核心实现解析 / 2. 多 LoRA 批处理调度): the batch is grouped
// by LoRA id so every group can be run contiguously with its own A, B.
//
// One CTA performs a stable counting sort of the token indices by adapter id.
// Key = id + 1 (key 0 collects the base-only tokens and any invalid id, so
// they come first). The tokens are cut into W contiguous chunks, one per warp
// (W = 32 when the per-(key, warp) counters fit in shared memory, else 8):
//   A. each warp counts its chunk per key (warp match, leader adds);
//   B. per-key warp prefixes + one block-wide exclusive scan over keys give
//      every (key, warp) its first output position, and every present key
//      >= 1 its segment (start, slot, prefix of 128-row units);
//   C. each warp walks its chunk again in token order and scatters; within a
//      32-token step equal keys are ranked by lane, so ties keep token order.
// The result is unique (a stable sort), so it is compared bit for bit.
//
// For pools of up to kSegMultiKeys keys, and for batches of kSegMultiMinT tokens and
// more, the same tables come from two kernels spread over the SMs (one CTA alone is
// bound by its own instruction issue):
//   1. seg_count_kernel, one CTA per kSegChunk tokens: keys, the chunk's per-key
//      counts, the per-tile adapter table and the zeroed shrink rows; the last CTA
//      to finish (an atomic ticket, nothing waits) turns the counts (chunk-major)
//      into each (key, chunk)'s first position by a scan over chunks -- a warp per
//      key when there are few keys, a thread per key otherwise -- and then over keys,
//      and writes the segment tables;
//   2. seg_scatter_kernel, one CTA per chunk: its warps place their tokens in turn,
//      ties ranked by lane, so the order is stable across and within chunks.
#include "device_common.cuh"

namespace lora {

namespace {

constexpr size_t kSegSmemLimit = 200 * 1024;

__device__ __forceinline__ uint32_t lanemask_lt()
{
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Key of a token; flags ids that are neither -1 nor a loaded slot.
__device__ __forceinline__ int token_key(int id, const PoolDev &pool, bool &bad)
{
    if (id == -1) return 0;
    if (slot_loaded(pool.slots, pool.slot_stride, pool.max_adapters, id)) return id + 1;
    bad = true;
    return 0;
}

template <int kSegWarps>
__global__ void __launch_bounds__(kSegWarps * 32, 1)
    seg_build_kernel(const int32_t *__restrict__ ids, int T, PoolDev pool, SegTables tabs,
                     int *__restrict__ err, int cache_keys, uint16_t *__restrict__ vhl, int ldh,
                     uint64_t *trace)
{
    constexpr int kSegThreads = kSegWarps * 32;
    trace_enter_released(trace);
    extern __shared__ uint32_t seg_smem[];
    const int K = pool.max_adapters + 1;
    uint32_t *cnt = seg_smem;                          // [K][kSegWarps]
    uint32_t *koff = seg_smem + (size_t)K * kSegWarps;  // [K]
    int *keys = reinterpret_cast<int *>(koff + K);      // [T] when cache_keys
    __shared__ uint32_t warp_tot[3][kSegWarps];
    __shared__ int any_bad;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int i = tid; i < K * kSegWarps; i += kSegThreads) cnt[i] = 0;
    if (tid == 0) any_bad = 0;
    bool bad = false;
    // keys computed once, by all threads in parallel, when they fit: each thread loads
    // kKeyBatch ids, then their slots' rank words, with all loads of a batch in flight
    // (two dependent round trips per batch instead of two per token)
    if (cache_keys) {
        constexpr int kKeyBatch = 8;
        for (int t0 = tid; t0 < T; t0 += kSegThreads * kKeyBatch) {
            int id[kKeyBatch], rk[kKeyBatch];
#pragma unroll
            for (int j = 0; j < kKeyBatch; ++j) {
                const int t = t0 + j * kSegThreads;
                id[j] = t < T ? ids[t] : -1;
            }
#pragma unroll
            for (int j = 0; j < kKeyBatch; ++j)
                rk[j] = (id[j] >= 0 && id[j] < pool.max_adapters)
                            ? pool.slots[(size_t)id[j] * pool.slot_stride + SLOT_RANK] : 0;
#pragma unroll
            for (int j = 0; j < kKeyBatch; ++j) {
                const int t = t0 + j * kSegThreads;
                if (t >= T) continue;
                int key = 0;  // as token_key: -1 -> 0, a loaded slot -> id + 1, else bad
                if (id[j] != -1) {
                    if (rk[j] > 0) key = id[j] + 1;
                    else bad = true;
                }
                keys[t] = key;
            }
        }
    }
    __syncthreads();

    const int chunk = (T + kSegWarps - 1) / kSegWarps;
    const int t0 = min(T, warp * chunk), t1 = min(T, t0 + chunk);

    // ---- A: per-warp counts; the shrink output rows of tokens without an adapter are
    // zeroed here (the prefill expand reads them inside single-adapter tiles)
    for (int base = t0; base < t1; base += 32) {
        const int t = base + lane;
        const bool valid = t < t1;
        int key = 0;
        if (valid) key = cache_keys ? keys[t] : token_key(ids[t], pool, bad);
        if (valid && key == 0 && vhl != nullptr) {
            uint4 *row = reinterpret_cast<uint4 *>(vhl + (size_t)t * ldh);
            for (int i = 0; i < ldh / 8; ++i) row[i] = make_uint4(0, 0, 0, 0);
        }
        const unsigned active = __ballot_sync(0xffffffffu, valid);
        if (valid) {
            const unsigned same = __match_any_sync(active, key);
            if (lane == __ffs(same) - 1) cnt[key * kSegWarps + warp] += __popc(same);
        }
    }
    if (bad) any_bad = 1;
    __syncthreads();

    // ---- B1: exclusive prefix over warps inside each key; koff = key total
    for (int k = tid; k < K; k += kSegThreads) {
        uint32_t run = 0;
#pragma unroll
        for (int w = 0; w < kSegWarps; ++w) {
            const uint32_t c = cnt[k * kSegWarps + w];
            cnt[k * kSegWarps + w] = run;
            run += c;
        }
        koff[k] = run;
    }
    __syncthreads();

    // ---- B2: block-wide exclusive scan over keys of (tokens, segments, units)
    const int per = (K + kSegThreads - 1) / kSegThreads;
    const int k_lo = min(K, tid * per), k_hi = min(K, k_lo + per);
    uint32_t sc = 0, ss = 0, su = 0;
    for (int k = k_lo; k < k_hi; ++k) {
        const uint32_t tot = koff[k];
        sc += tot;
        if (k >= 1 && tot > 0) {
            ss += 1;
            su += (tot + kShrinkRows - 1) / kShrinkRows;
        }
    }
    uint32_t ic = sc, is = ss, iu = su;  // inclusive warp scan
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t c = __shfl_up_sync(0xffffffffu, ic, o);
        const uint32_t s = __shfl_up_sync(0xffffffffu, is, o);
        const uint32_t u = __shfl_up_sync(0xffffffffu, iu, o);
        if (lane >= o) {
            ic += c;
            is += s;
            iu += u;
        }
    }
    if (lane == 31) {
        warp_tot[0][warp] = ic;
        warp_tot[1][warp] = is;
        warp_tot[2][warp] = iu;
    }
    __syncthreads();
    uint32_t wc = 0, ws = 0, wu = 0, all_s = 0, all_u = 0;
    for (int w = 0; w < kSegWarps; ++w) {
        if (w < warp) {
            wc += warp_tot[0][w];
            ws += warp_tot[1][w];
            wu += warp_tot[2][w];
        }
        all_s += warp_tot[1][w];
        all_u += warp_tot[2][w];
    }
    uint32_t pc = wc + ic - sc, ps = ws + is - ss, pu = wu + iu - su;  // exclusive
    if (tid == 0) tabs.hdr[HDR_NBASE] = (int32_t)koff[0];
    __syncthreads();  // koff[0] read above before it is overwritten below
    for (int k = k_lo; k < k_hi; ++k) {
        const uint32_t tot = koff[k];
        koff[k] = pc;
        if (k >= 1 && tot > 0) {
            tabs.seg_start[ps] = (int32_t)pc;
            tabs.seg_slot[ps] = k - 1;
            tabs.seg_ublk[ps] = (int32_t)pu;
            ps += 1;
            pu += (tot + kShrinkRows - 1) / kShrinkRows;
        }
        pc += tot;
    }
    if (tid == 0) {
        tabs.hdr[HDR_NUMSEG] = (int32_t)all_s;
        tabs.hdr[HDR_UNITS] = (int32_t)all_u;
        tabs.seg_start[all_s] = T;
        tabs.seg_ublk[all_s] = (int32_t)all_u;
        if (any_bad) atomicOr(err, kErrBadIdBit);
    }
    __syncthreads();

    // ---- C: stable scatter
    for (int base = t0; base < t1; base += 32) {
        const int t = base + lane;
        const bool valid = t < t1;
        bool unused = false;
        int key = 0;
        if (valid) key = cache_keys ? keys[t] : token_key(ids[t], pool, unused);
        const unsigned active = __ballot_sync(0xffffffffu, valid);
        if (valid) {
            const unsigned same = __match_any_sync(active, key);
            const uint32_t pos =
                koff[key] + cnt[key * kSegWarps + warp] + __popc(same & lanemask_lt());
#ifdef LORA_CHECK
            if (check_range((int)pos, 0, T, err))
#endif
                tabs.order[pos] = t;
            __syncwarp(active);
            if (lane == __ffs(same) - 1) cnt[key * kSegWarps + warp] += __popc(same);
        }
        __syncwarp();
    }

    // ---- D: adapters of each 128-token tile (in token order), for the prefill GEMM
    const int ntile = (T + 127) / 128;
    for (int tile = warp; tile < ntile; tile += kSegWarps) {
        int lo = 0x7fffffff, hi = -1;
        for (int i = lane; i < 128; i += 32) {
            const int t = tile * 128 + i;
            if (t < T) {
                bool unused = false;
                const int key = cache_keys ? keys[t] : token_key(ids[t], pool, unused);
                if (key > 0) {
                    lo = min(lo, key - 1);
                    hi = max(hi, key - 1);
                }
            }
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
            hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
        }
        if (lane == 0) tabs.tile_info[tile] = hi < 0 ? kTileNoAdapter : (lo == hi ? hi : kTileMixed);
    }
    if (trace) {
        __syncthreads();
        trace_exit(trace);
    }
}

// ------------------------------------------------------- multi-CTA builder

// Exclusive scan of (tokens, segments, 128-row units) over the K keys by all
// kSegChunk threads of the CTA, key 0 (base only) forming no segment; the segment
// tables and the header are written, and `first` receives each key's first position.
__device__ __forceinline__ void scan_keys(const int *total, int K, int T, SegTables tabs, int *first)
{
    constexpr int kWarps = kSegChunk / 32;
    __shared__ uint32_t warp_tot[3][kWarps];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int per = (K + kSegChunk - 1) / kSegChunk;
    const int k_lo = min(K, tid * per), k_hi = min(K, k_lo + per);
    uint32_t sc = 0, ss = 0, su = 0;
    for (int k = k_lo; k < k_hi; ++k) {
        const uint32_t tot = (uint32_t)total[k];
        sc += tot;
        if (k >= 1 && tot > 0) {
            ss += 1;
            su += (tot + kShrinkRows - 1) / kShrinkRows;
        }
    }
    uint32_t ic = sc, is = ss, iu = su;  // inclusive warp scan
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t c = __shfl_up_sync(0xffffffffu, ic, o);
        const uint32_t v = __shfl_up_sync(0xffffffffu, is, o);
        const uint32_t u = __shfl_up_sync(0xffffffffu, iu, o);
        if (lane >= o) {
            ic += c;
            is += v;
            iu += u;
        }
    }
    if (lane == 31) {
        warp_tot[0][warp] = ic;
        warp_tot[1][warp] = is;
        warp_tot[2][warp] = iu;
    }
    __syncthreads();
    uint32_t wc = 0, ws = 0, wu = 0, all_s = 0, all_u = 0;
    for (int w = 0; w < kWarps; ++w) {
        if (w < warp) {
            wc += warp_tot[0][w];
            ws += warp_tot[1][w];
            wu += warp_tot[2][w];
        }
        all_s += warp_tot[1][w];
        all_u += warp_tot[2][w];
    }
    uint32_t pc = wc + ic - sc, ps = ws + is - ss, pu = wu + iu - su;  // exclusive
    for (int k = k_lo; k < k_hi; ++k) {
        const uint32_t tot = (uint32_t)total[k];
        first[k] = (int)pc;
        if (k >= 1 && tot > 0) {
            tabs.seg_start[ps] = (int32_t)pc;
            tabs.seg_slot[ps] = k - 1;
            tabs.seg_ublk[ps] = (int32_t)pu;
            ps += 1;
            pu += (tot + kShrinkRows - 1) / kShrinkRows;
        }
        pc += tot;
    }
    if (tid == 0) {
        tabs.hdr[HDR_NBASE] = total[0];
        tabs.hdr[HDR_NUMSEG] = (int32_t)all_s;
        tabs.hdr[HDR_UNITS] = (int32_t)all_u;
        tabs.seg_start[all_s] = T;
        tabs.seg_ublk[all_s] = (int32_t)all_u;
    }
}

__global__ void __launch_bounds__(kSegChunk)
    seg_count_kernel(const int32_t *__restrict__ ids, int T, PoolDev pool, SegTables tabs,
                     int *__restrict__ err, uint16_t *__restrict__ vhl, int ldh, uint64_t *trace)
{
    trace_enter_released(trace);
    constexpr int kWarps = kSegChunk / 32;
    extern __shared__ int hist[];  // [K]: this chunk's counts, then (last CTA) the totals
    __shared__ int lo_w[kWarps], hi_w[kWarps];
    __shared__ int is_last;
    const int K = pool.max_adapters + 1, chunks = (int)gridDim.x;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int k = tid; k < K; k += kSegChunk) hist[k] = 0;
    __syncthreads();

    const int t = (int)blockIdx.x * kSegChunk + tid;
    bool bad = false;
    int key = -1;
    if (t < T) {
        key = token_key(ids[t], pool, bad);
        tabs.keys[t] = key;
        atomicAdd(&hist[key], 1);
        if (key == 0 && vhl != nullptr) {  // the expand reads these rows inside one-adapter tiles
            uint4 *row = reinterpret_cast<uint4 *>(vhl + (size_t)t * ldh);
            for (int i = 0; i < ldh / 8; ++i) row[i] = make_uint4(0, 0, 0, 0);
        }
    }
    if (bad) atomicOr(err, kErrBadIdBit);
    // adapters of the chunk's two 128-token tiles (four warps each)
    int lo = key > 0 ? key - 1 : 0x7fffffff, hi = key > 0 ? key - 1 : -1;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
        hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    if (lane == 0) {
        lo_w[warp] = lo;
        hi_w[warp] = hi;
    }
    __syncthreads();
    if (tid < kSegChunk / 128) {
        const int tile = (int)blockIdx.x * (kSegChunk / 128) + tid;
        if (tile * 128 < T) {
            int l = 0x7fffffff, h = -1;
            for (int w = tid * 4; w < tid * 4 + 4; ++w) {
                l = min(l, lo_w[w]);
                h = max(h, hi_w[w]);
            }
            tabs.tile_info[tile] = h < 0 ? kTileNoAdapter : (l == h ? h : kTileMixed);
        }
    }
    for (int k = tid; k < K; k += kSegChunk) tabs.chist[(size_t)blockIdx.x * K + k] = hist[k];

    // the last chunk to finish turns the counts into positions
    __threadfence();
    __syncthreads();
    if (tid == 0) is_last = atomicAdd(tabs.ticket, 1) == chunks - 1;
    __syncthreads();
    if (!is_last) {
        trace_exit(trace);
        return;
    }
    __threadfence();
    // per key: exclusive scan over the chunks, the key's total into hist[]. Few keys
    // (a prefill of a few long sequences): a warp per key, 32 chunks per step; many
    // keys: a thread per key, its 16 chunks' loads issued together (the counts are
    // chunk-major, so they are coalesced across the CTA)
    if (K <= 2 * kWarps) {
        for (int k = warp; k < K; k += kWarps) {
            int carry = 0;
            for (int c0 = 0; c0 < chunks; c0 += 32) {
                const int c = c0 + lane;
                const int v = c < chunks ? __ldcg(tabs.chist + (size_t)c * K + k) : 0;
                int inc = v;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int n = __shfl_up_sync(0xffffffffu, inc, o);
                    if (lane >= o) inc += n;
                }
                if (c < chunks) tabs.chist[(size_t)c * K + k] = carry + inc - v;
                carry += __shfl_sync(0xffffffffu, inc, 31);
            }
            if (lane == 0) hist[k] = carry;
        }
    } else for (int k = tid; k < K; k += 2 * kSegChunk) {
        // two keys per thread (k and k + kSegChunk): 32 loads in flight per round
        const int k2 = k + kSegChunk;
        const bool two = k2 < K;
        int carry = 0, carry2 = 0;
        for (int c0 = 0; c0 < chunks; c0 += 16) {
            int v[16], v2[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                v[i] = c0 + i < chunks ? __ldcg(tabs.chist + (size_t)(c0 + i) * K + k) : 0;
                v2[i] = two && c0 + i < chunks ? __ldcg(tabs.chist + (size_t)(c0 + i) * K + k2) : 0;
            }
#pragma unroll
            for (int i = 0; i < 16; ++i)
                if (c0 + i < chunks) {
                    tabs.chist[(size_t)(c0 + i) * K + k] = carry;
                    carry += v[i];
                    if (two) {
                        tabs.chist[(size_t)(c0 + i) * K + k2] = carry2;
                        carry2 += v2[i];
                    }
                }
        }
        hist[k] = carry;
        if (two) hist[k2] = carry2;
    }
    __syncthreads();
    scan_keys(hist, K, T, tabs, tabs.chist + (size_t)K * chunks);
    if (tid == 0) *tabs.ticket = 0;  // for the next call (after this kernel completes)
    __syncthreads();
    trace_exit(trace);
}

__global__ void __launch_bounds__(kSegChunk)
    seg_scatter_kernel(int T, int K, SegTables tabs, int *err, uint64_t *trace)
{
    trace_enter_released(trace);
    constexpr int kWarps = kSegChunk / 32;
    extern __shared__ int run[];  // [K] the next position of each key in this chunk
    const int chunks = (int)gridDim.x;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int32_t *first = tabs.chist + (size_t)K * chunks;
    for (int k = tid; k < K; k += kSegChunk) run[k] = first[k] + tabs.chist[(size_t)blockIdx.x * K + k];
    const int t = (int)blockIdx.x * kSegChunk + tid;
    const int key = t < T ? tabs.keys[t] : 0;
    __syncthreads();
    // warps in turn (token order), lanes ranked within a warp: a stable order
    for (int w = 0; w < kWarps; ++w) {
        if (warp == w) {
            const unsigned active = __ballot_sync(0xffffffffu, t < T);
            if (t < T) {
                const unsigned same = __match_any_sync(active, key);
                const int pos = run[key] + __popc(same & lanemask_lt());
#ifdef LORA_CHECK
                if (check_range(pos, 0, T, err))
#endif
                    tabs.order[pos] = t;
                __syncwarp(active);
                if (lane == __ffs(same) - 1) run[key] += __popc(same);
            }
        }
        __syncthreads();
    }
    trace_exit(trace);
}

}  // namespace

size_t seg_build_smem_bytes(int max_adapters, int warps)
{
    const size_t K = (size_t)max_adapters + 1;
    return K * warps * sizeof(uint32_t) + K * sizeof(uint32_t);
}

namespace {

template <int W>
cudaError_t launch_seg_build_w(const int32_t *ids, int T, const PoolDev &pool, SegTables tabs, int *err,
                               uint16_t *vhl, int ldh, cudaStream_t stream, uint64_t *trace)
{
    size_t smem = seg_build_smem_bytes(pool.max_adapters, W);
    const int cache_keys = smem + (size_t)T * sizeof(int) <= kSegSmemLimit;
    if (cache_keys) smem += (size_t)T * sizeof(int);
    cudaError_t e = ensure_smem_attr((const void *)seg_build_kernel<W>, smem);
    if (e != cudaSuccess) return e;
    seg_build_kernel<W><<<1, W * 32, smem, stream>>>(ids, T, pool, tabs, err, cache_keys, vhl, ldh, trace);
    return cudaGetLastError();
}

}  // namespace

// 32 warps (each walks a 32nd of the tokens) when their counters and the cached keys
// fit in shared memory; 8 warps otherwise (large pools).
cudaError_t launch_seg_build(const int32_t *ids, int T, const PoolDev &pool, SegTables tabs,
                             int *err, uint16_t *vhl, int ldh, cudaStream_t stream, uint64_t *trace)
{
    const int K = pool.max_adapters + 1;
    if (tabs.chist != nullptr && K <= kSegMultiMaxKeys && (K <= kSegMultiKeys || T >= kSegMultiMinT)) {
        const int chunks = (T + kSegChunk - 1) / kSegChunk;
        const size_t smem = (size_t)K * sizeof(int);
        cudaError_t e = ensure_smem_attr((const void *)seg_count_kernel, smem);
        if (e == cudaSuccess) e = ensure_smem_attr((const void *)seg_scatter_kernel, smem);
        if (e != cudaSuccess) return e;
        seg_count_kernel<<<chunks, kSegChunk, smem, stream>>>(ids, T, pool, tabs, err, vhl, ldh, trace);
        seg_scatter_kernel<<<chunks, kSegChunk, smem, stream>>>(T, K, tabs, err, trace);
        return cudaGetLastError();
    }
    if (seg_build_smem_bytes(pool.max_adapters, 32) + (size_t)T * sizeof(int) <= kSegSmemLimit)
        return launch_seg_build_w<32>(ids, T, pool, tabs, err, vhl, ldh, stream, trace);
    return launch_seg_build_w<8>(ids, T, pool, tabs, err, vhl, ldh, stream, trace);
}

}  // namespace lora
