// pool.cu -- host runtime behind the C ABI: the paged adapter pool, the slot
// table, scratch management and the kernel sequence of one lora_linear call.
//
// The pool follows the unified adapter memory pool of the vLLM tutorial
// ("vLLM 的 Multi-LoRA 怎么实现", item 1) and the LoRA-Land blog's hot-plug API
// (核心实现解析 / 3: load_adapter moves A,B to the GPU and indexes them;
// unload_adapter releases them). Pages hold 8 rank rows; the arenas are
// allocated once at creation, so load and unload only move pages between a
// free list and the slot table and never allocate.
#include <algorithm>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <map>
#include <vector>

#include <cudaTypedefs.h>

#include "../../include/lora_linear.h"
#include "device_common.cuh"
#include "pool_state.h"

using namespace lora;

namespace lora {

lora_status alloc_dev(lora_pool *p, void **ptr, size_t bytes)
{
    if (bytes == 0) bytes = 16;
    if (cudaMalloc(ptr, bytes) != cudaSuccess) {
        cudaGetLastError();
        *ptr = nullptr;
        return LORA_ERR_OOM;
    }
    p->bytes_held += bytes;
    return LORA_OK;
}

void free_dev(lora_pool *p, void *ptr, size_t bytes)
{
    if (ptr) {
        cudaFree(ptr);
        p->bytes_held -= bytes ? bytes : 16;
    }
}

PoolDev pool_view(const lora_pool *p)
{
    PoolDev v;
    v.A_pages = p->A_pages;
    v.B_pages = p->B_pages;
    v.slots = p->d_slots;
    v.slot_stride = p->slot_stride;
    v.max_adapters = p->max_adapters;
    v.max_pages = p->max_pages;
    v.num_pages = p->num_pages;
    v.d_in = p->d_in;
    v.d_out = p->d_out;
    return v;
}

lora_status order_after_changes(lora_pool *p, cudaStream_t stream)
{
    if (p->copy_epoch == p->waited_epoch && stream == p->waited_stream) return LORA_OK;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    CUDA_TRY(cudaStreamIsCapturing(stream, &cs));
    if (cs != cudaStreamCaptureStatusNone) return LORA_OK;  // graph replays are the caller's order
    CUDA_TRY(cudaStreamWaitEvent(stream, p->ev_copy, 0));
    p->waited_epoch = p->copy_epoch;
    p->waited_stream = stream;
    return LORA_OK;
}

lora_status note_call(lora_pool *p, cudaStream_t stream)
{
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    CUDA_TRY(cudaStreamIsCapturing(stream, &cs));
    if (cs != cudaStreamCaptureStatusNone) return LORA_OK;  // graph replays are the caller's order
    // every later change on the copy stream (pages, table rows, the error-word read)
    // starts after this call, whichever stream it ran on
    CUDA_TRY(cudaEventRecord(p->ev_call, stream));
    CUDA_TRY(cudaStreamWaitEvent(p->copy_stream, p->ev_call, 0));
    return LORA_OK;
}

lora_status stage_row_ready(lora_pool *p, int slot, int32_t **row)
{
    *row = p->stage_rows + (size_t)slot * (p->slot_stride + p->max_pages);
    if (slot < p->max_adapters) CUDA_TRY(cudaEventSynchronize(p->slot_copy_ev[slot]));
    return LORA_OK;
}

lora_status enqueue_row(lora_pool *p, int slot, const int32_t *row)
{
    cudaStream_t s = p->copy_stream;
    CUDA_TRY(cudaMemcpyAsync(p->d_slots + (size_t)slot * p->slot_stride, row,
                             sizeof(int32_t) * p->slot_stride, cudaMemcpyHostToDevice, s));
    if (row != p->stage_rows + (size_t)p->max_adapters * (p->slot_stride + p->max_pages))
        CUDA_TRY(cudaEventRecord(p->slot_copy_ev[slot], s));
    CUDA_TRY(cudaEventRecord(p->ev_copy, s));
    p->copy_epoch += 1;
    return LORA_OK;
}

lora_status release_pages(lora_pool *p, const int32_t *pages, int n)
{
    if (n <= 0) return LORA_OK;
    cudaEvent_t ev = nullptr;
    if (!p->idle_events.empty()) {
        ev = p->idle_events.back();
        p->idle_events.pop_back();
    } else {
        CUDA_TRY(cudaEventCreateWithFlags(&ev, cudaEventDisableTiming));
    }
    if (cudaEventRecord(ev, p->copy_stream) != cudaSuccess) {
        cudaGetLastError();
        cudaEventDestroy(ev);
        return LORA_ERR_CUDA;  // the pages stay out of the free list
    }
    p->freed.push_back({ev, std::vector<int32_t>(pages, pages + n)});
    return LORA_OK;
}

// Freed batches whose event has completed join the free list (the batches were
// recorded in order on one stream, so the first pending one ends the scan).
static void reclaim_pages(lora_pool *p)
{
    while (!p->freed.empty()) {
        lora_pool::FreedBatch &b = p->freed.front();
        const cudaError_t q = cudaEventQuery(b.ev);
        if (q != cudaSuccess) {
            if (q != cudaErrorNotReady) cudaGetLastError();
            break;
        }
        p->free_pages.insert(p->free_pages.end(), b.pages.rbegin(), b.pages.rend());
        p->idle_events.push_back(b.ev);
        p->freed.pop_front();
    }
}

int free_page_count(const lora_pool *p)
{
    size_t n = p->free_pages.size();
    for (const lora_pool::FreedBatch &b : p->freed) n += b.pages.size();
    return (int)n;
}

void take_pages(lora_pool *p, int n, int32_t *out, bool *fresh)
{
    reclaim_pages(p);
    *fresh = (int)p->free_pages.size() >= n;
    int k = 0;
    while (k < n && !p->free_pages.empty()) {
        out[k++] = p->free_pages.back();
        p->free_pages.pop_back();
    }
    // not enough: the oldest freed pages, written on the copy stream after the calls
    while (k < n && !p->freed.empty()) {
        lora_pool::FreedBatch &b = p->freed.front();
        while (k < n && !b.pages.empty()) {
            out[k++] = b.pages.back();
            b.pages.pop_back();
        }
        if (b.pages.empty()) {
            p->idle_events.push_back(b.ev);  // a later record replaces its pending one
            p->freed.pop_front();
        }
    }
}

}  // namespace lora

namespace {

size_t seg_entries(const lora_pool *p, int T) { return (size_t)std::min(T, p->max_adapters) + 1; }

// The multi-CTA segment builder's count table: (chunk, key) counts, then one row of
// first positions (pools of up to kSegMultiMaxKeys keys; else 0: not used).
size_t seg_chist_ints(const lora_pool *p, int T)
{
    const size_t K = (size_t)p->max_adapters + 1;
    if (K > (size_t)kSegMultiMaxKeys) return 0;
    return K * ((size_t)(T + kSegChunk - 1) / kSegChunk + 1);
}

void free_scratch(lora_pool *p)
{
    const int T = p->cap_T;
    if (T == 0) return;
    free_dev(p, p->order, sizeof(int32_t) * T);
    free_dev(p, p->hdr, sizeof(int32_t) * 4);
    free_dev(p, p->seg_start, sizeof(int32_t) * seg_entries(p, T));
    free_dev(p, p->seg_slot, sizeof(int32_t) * seg_entries(p, T));
    free_dev(p, p->seg_ublk, sizeof(int32_t) * seg_entries(p, T));
    free_dev(p, p->tile_info, sizeof(int32_t) * (size_t)((T + 127) / 128));
    p->tile_info = nullptr;
    free_dev(p, p->seg_keys, sizeof(int32_t) * T);
    free_dev(p, p->seg_chist, sizeof(int32_t) * seg_chist_ints(p, T));
    free_dev(p, p->seg_ticket, sizeof(int32_t));
    p->seg_keys = p->seg_chist = p->seg_ticket = nullptr;
    free_dev(p, p->V, sizeof(float) * (size_t)T * p->ldv);
    free_dev(p, p->Vhl, sizeof(uint16_t) * (size_t)T * p->ldh);
    p->Vhl = nullptr;
    free_dev(p, p->partials, sizeof(float) * p->partials_floats);
    p->order = p->hdr = p->seg_start = p->seg_slot = p->seg_ublk = nullptr;
    p->V = p->partials = nullptr;
    p->partials_floats = 0;
    p->cap_T = 0;
}

lora_status ensure_scratch(lora_pool *p, int T)
{
    if (T <= p->cap_T) return LORA_OK;
    CUDA_TRY(cudaDeviceSynchronize());  // earlier calls may still read the old scratch
    free_scratch(p);
    const size_t se = seg_entries(p, T);
    DecodePlan plan;
    if (!plan_decode(1, std::max(1, std::min(T, kDecodeMaxT)), &p->d_in, &p->d_out, &p->max_pages,
                     p->num_sms, &plan))
        return LORA_ERR_SHAPE;
    const size_t pf = std::max(decode_partials_floats(plan), p->partials_floats);
    lora_status st;
    if ((st = alloc_dev(p, (void **)&p->order, sizeof(int32_t) * T)) ||
        (st = alloc_dev(p, (void **)&p->hdr, sizeof(int32_t) * 4)) ||
        (st = alloc_dev(p, (void **)&p->seg_start, sizeof(int32_t) * se)) ||
        (st = alloc_dev(p, (void **)&p->seg_slot, sizeof(int32_t) * se)) ||
        (st = alloc_dev(p, (void **)&p->seg_ublk, sizeof(int32_t) * se)) ||
        (st = alloc_dev(p, (void **)&p->tile_info, sizeof(int32_t) * (size_t)((T + 127) / 128))) ||
        (st = alloc_dev(p, (void **)&p->V, sizeof(float) * (size_t)T * p->ldv)) ||
        (st = alloc_dev(p, (void **)&p->Vhl, sizeof(uint16_t) * (size_t)T * p->ldh)) ||
        (st = alloc_dev(p, (void **)&p->partials, sizeof(float) * pf))) {
        p->cap_T = T;
        p->partials_floats = pf;
        free_scratch(p);
        return st;
    }
    p->cap_T = T;
    p->partials_floats = pf;
    if (seg_chist_ints(p, T) > 0) {
        if ((st = alloc_dev(p, (void **)&p->seg_keys, sizeof(int32_t) * T)) ||
            (st = alloc_dev(p, (void **)&p->seg_chist, sizeof(int32_t) * seg_chist_ints(p, T))) ||
            (st = alloc_dev(p, (void **)&p->seg_ticket, sizeof(int32_t)))) {
            free_scratch(p);
            return st;
        }
        CUDA_TRY(cudaMemset(p->seg_ticket, 0, sizeof(int32_t)));
    }
    return LORA_OK;
}

SegTables seg_tables(const lora_pool *p)
{
    SegTables t;
    t.order = p->order;
    t.hdr = p->hdr;
    t.seg_start = p->seg_start;
    t.seg_slot = p->seg_slot;
    t.seg_ublk = p->seg_ublk;
    t.tile_info = p->tile_info;
    t.keys = p->seg_keys;
    t.chist = p->seg_chist;
    t.ticket = p->seg_ticket;
    return t;
}

// Tensor maps are pure host descriptors of (pointer, shape, box); a small
// per-pool cache avoids re-encoding them on every call with the same buffers. The map
// is copied out: a later lookup of the same call may reuse the cache entry.
bool tmap_for(lora_pool *p, CUtensorMap *out, const void *base, uint64_t inner, uint64_t rows,
              uint32_t box_inner, uint32_t box_rows)
{
    for (auto &e : p->tmaps)
        if (e.base == base && e.inner == inner && e.rows == rows && e.box_inner == box_inner &&
            e.box_rows == box_rows) {
            *out = e.map;
            return true;
        }
    TmapEntry &e = p->tmaps[p->tmap_next];
    p->tmap_next = (p->tmap_next + 1) % (int)(sizeof(p->tmaps) / sizeof(p->tmaps[0]));
    e.base = nullptr;
    if (!make_tmap_bf16_2d(&e.map, base, inner, rows, inner * 2, box_inner, box_rows)) return false;
    e.base = base;
    e.inner = inner;
    e.rows = rows;
    e.box_inner = box_inner;
    e.box_rows = box_rows;
    *out = e.map;
    return true;
}

__global__ void pack_adapter_kernel(const uint16_t *__restrict__ A, const uint16_t *__restrict__ B,
                                    int rank, const int32_t *__restrict__ pages, int npages, int d_in,
                                    int d_out, uint16_t *__restrict__ A_pages,
                                    uint16_t *__restrict__ B_pages, int num_pages, int *err)
{
    const size_t totA = (size_t)npages * kRankPage * d_in;
    const size_t totB = (size_t)npages * d_out * kRankPage;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < totA + totB;
         i += (size_t)gridDim.x * blockDim.x) {
        if (i < totA) {
            const size_t per_page = (size_t)kRankPage * d_in;
            const int q = (int)(i / per_page);
            const size_t rem = i % per_page;
            const int jj = (int)(rem / d_in), k = (int)(rem % d_in);
            const int j = q * kRankPage + jj;
#ifdef LORA_CHECK
            if (!check_range(pages[q], 1, num_pages, err)) continue;  // never the zero page
#endif
            A_pages[(size_t)pages[q] * per_page + rem] = (j < rank) ? A[(size_t)k * rank + j] : 0;
        } else {
            const size_t i2 = i - totA;
            const size_t per_page = (size_t)d_out * kRankPage;
            const int q = (int)(i2 / per_page);
            const size_t rem = i2 % per_page;
            const int n = (int)(rem / kRankPage), jj = (int)(rem % kRankPage);
            const int j = q * kRankPage + jj;
#ifdef LORA_CHECK
            if (!check_range(pages[q], 1, num_pages, err)) continue;
#endif
            B_pages[(size_t)pages[q] * per_page + rem] = (j < rank) ? B[(size_t)j * d_out + n] : 0;
        }
    }
}

bool dims_ok(int d) { return d > 0 && d <= LORA_MAX_DIM && d % 8 == 0; }

// One bounded wait on an mbarrier that nothing arrives on: the kernels' wait
// runs out after limit_ns, raises the timeout bit and returns (no trap, no hang).
__global__ void wait_selftest_kernel(int *err, uint64_t limit_ns)
{
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait(&bar, 0, &abort_flag, err, limit_ns);
    __syncthreads();
}

// err[1] = the error word err[0], which is cleared in the same atomic step.
__global__ void read_clear_kernel(int *err) { err[1] = atomicExch(err, 0); }

// A producer of the kind that programmatic dependent launch allows: it lets the next
// kernel in the stream start at once, then, after `delay_ns`, writes dst. Anything
// that reads dst before its own wait on this kernel sees the old values.
__global__ void delayed_copy_kernel(const int32_t *src, int32_t *dst, int n, uint64_t delay_ns)
{
    pdl_launch_dependents();
    if (threadIdx.x == 0) {
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < delay_ns) {
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += blockDim.x) dst[i] = src[i];
}

// Split-K partials of a grouped decode call (held by its first pool): grown on
// first use of a larger group, like the rest of the scratch.
lora_status ensure_partials(lora_pool *p, size_t floats)
{
    if (floats <= p->partials_floats) return LORA_OK;
    CUDA_TRY(cudaDeviceSynchronize());  // earlier calls may still read the old buffer
    free_dev(p, p->partials, sizeof(float) * p->partials_floats);
    p->partials = nullptr;
    p->partials_floats = 0;
    lora_status st = alloc_dev(p, (void **)&p->partials, sizeof(float) * floats);
    if (st == LORA_OK) p->partials_floats = floats;
    return st;
}

// Measurement hook of one call: event k+1 closes kernel slot k (inside a graph
// capture the records become event nodes replayed with the graph).
struct CallMarks {
    lora_pool *p;
    cudaStream_t stream;
    cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
    bool begin()
    {
        if (!p->timing) return true;
        for (bool &u : p->ev_used) u = false;
        if (cudaStreamIsCapturing(stream, &capture) != cudaSuccess) return false;
        return mark(-1);
    }
    bool mark(int slot)
    {
        if (!p->timing) return true;
        if (slot >= 0) p->ev_used[slot] = true;
        p->ev_last = slot + 1;
        const unsigned flags =
            capture == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : cudaEventRecordDefault;
        return cudaEventRecordWithFlags(p->ev[slot + 1], stream, flags) == cudaSuccess;
    }
};

// The decode path for n problems that share the ids (scratch already sized for T
// on every pool). Per-token (BGMV-style) shrink fused into the GEMM kernel: no
// segment tables.
// The span-trace words of the next call on p (LORA_KERNEL_SLOTS x kTraceWords), or nullptr.
uint64_t *next_trace(lora_pool *p)
{
    if (!p->trace) return nullptr;
    uint64_t *t = p->trace + (size_t)(p->trace_k % p->trace_calls) * LORA_KERNEL_SLOTS * kTraceWords;
    p->trace_k += 1;
    return t;
}

uint64_t *trace_slot(uint64_t *t, int slot) { return t ? t + kTraceWords * slot : nullptr; }

lora_status run_decode(lora_pool *const *pools, int n, const void *const *X, const void *const *W,
                       const int32_t *ids, int T, void *const *Y, cudaStream_t stream, bool with_lora,
                       CallMarks &marks)
{
    lora_pool *p0 = pools[0];
    int d_in[kMaxGroup], d_out[kMaxGroup], pages[kMaxGroup];
    for (int m = 0; m < n; ++m) {
        d_in[m] = pools[m]->d_in;
        d_out[m] = pools[m]->d_out;
        pages[m] = with_lora ? pools[m]->max_pages : 0;
    }
    DecodePlan plan;
    if (!plan_decode(n, T, d_in, d_out, pages, p0->num_sms, &plan)) return LORA_ERR_SHAPE;
    lora_status st = ensure_partials(p0, decode_partials_floats(plan));
    if (st != LORA_OK) return st;
    DecodeMaps maps;
    for (int m = 0; m < n; ++m) {
        lora_pool *p = pools[m];
        if (!tmap_for(p, &maps.W[m], W[m], p->d_in, p->d_out, 64, 128) ||
            !tmap_for(p, &maps.X[m], X[m], p->d_in, T, 64, plan.ntok))
            return LORA_ERR_ARG;
        DecodeProblem &q = plan.prob[m];
        q.pool = pool_view(p);
        q.X = static_cast<const uint16_t *>(X[m]);
        q.V = p->V;
        q.ldv = p->ldv;
        q.Y = static_cast<uint16_t *>(Y[m]);
        q.err = p->d_err;
    }
    const int32_t *tids = with_lora ? ids : nullptr;
    plan.trace = next_trace(p0);
    CUDA_TRY(launch_gemm_decode(maps, plan, tids, p0->partials, p0->d_err, stream));
    if (!marks.mark(2)) return LORA_ERR_CUDA;
    CUDA_TRY(launch_finish_decode(plan, p0->partials, tids, stream));
    if (!marks.mark(3)) return LORA_ERR_CUDA;
    return LORA_OK;
}

lora_status run_linear(lora_pool *p, const void *X, const void *W, const int32_t *ids, int T,
                       void *Y, cudaStream_t stream, bool with_lora);

// The layer over a 4-bit base: decode-sized batches run the GEMM kernel that
// dequantises W tiles in shared memory; larger ones dequantise W into pool scratch and
// run the bf16 prefill path.
lora_status run_linear_q4(lora_pool *p, const void *X, const void *Wq, const void *S, const void *Z,
                          const int32_t *ids, int T, void *Y, cudaStream_t stream, bool with_lora)
{
    if (!p || !X || !Wq || !S || !Z || !Y || (with_lora && !ids) || T < 0) return LORA_ERR_ARG;
    if (p->d_in % kQ4Group != 0 || p->d_out % 16 != 0) return LORA_ERR_SHAPE;
    if (((uintptr_t)Wq | (uintptr_t)S | (uintptr_t)Z) & 15) return LORA_ERR_ARG;  // 16-byte loads
    int path = p->path;
    if (path == LORA_PATH_AUTO) path = T <= kDecodeMaxT ? LORA_PATH_DECODE : LORA_PATH_PREFILL;
    if (path == LORA_PATH_DECODE && T > kDecodeMaxT) return LORA_ERR_ARG;
    if (T == 0) return LORA_OK;
    if (path == LORA_PATH_PREFILL) {
        if (!p->wdq) {
            lora_status st = alloc_dev(p, (void **)&p->wdq, (size_t)p->d_out * p->d_in * 2);
            if (st != LORA_OK) return st;
        }
        CUDA_TRY(launch_dequant_q4(static_cast<const uint8_t *>(Wq), static_cast<const uint16_t *>(S),
                                   static_cast<const uint8_t *>(Z), p->d_out, p->d_in, p->wdq, stream));
        return run_linear(p, X, p->wdq, ids, T, Y, stream, with_lora);
    }
    lora_status st = ensure_scratch(p, T);
    if (st == LORA_OK) st = order_after_changes(p, stream);
    if (st != LORA_OK) return st;
    const int no_pages = 0;
    DecodePlan plan;
    if (!plan_decode(1, T, &p->d_in, &p->d_out, with_lora ? &p->max_pages : &no_pages, p->num_sms, &plan))
        return LORA_ERR_SHAPE;
    plan.prob[0].pool = pool_view(p);
    if (!plan_decode_q4(&plan)) return LORA_ERR_SHAPE;
    if ((st = ensure_partials(p, decode_partials_floats(plan))) != LORA_OK) return st;
    DecodeMapsQ4 maps;
    const int groups = p->d_in / kQ4Group;
    if (!make_tmap_u8_2d(&maps.Wq, Wq, p->d_in / 2, p->d_out, p->d_in / 2, 64, 128) ||
        !make_tmap_bf16_2d(&maps.S, S, p->d_out, groups, (uint64_t)p->d_out * 2, 128, 1, false) ||
        !make_tmap_u8_2d(&maps.Z, Z, p->d_out, groups, p->d_out, 128, 1) ||
        !make_tmap_bf16_2d(&maps.X, X, p->d_in, T, (uint64_t)p->d_in * 2, 64, plan.ntok))
        return LORA_ERR_ARG;
    DecodeProblem &q = plan.prob[0];
    q.X = static_cast<const uint16_t *>(X);
    q.V = p->V;
    q.ldv = p->ldv;
    q.Y = static_cast<uint16_t *>(Y);
    q.err = p->d_err;
    plan.trace = next_trace(p);
    const int32_t *tids = with_lora ? ids : nullptr;
    CallMarks marks{p, stream};
    if (!marks.begin()) return LORA_ERR_CUDA;
    CUDA_TRY(launch_gemm_decode_q4(maps, plan, tids, p->partials, p->d_err, stream));
    if (!marks.mark(2)) return LORA_ERR_CUDA;
    CUDA_TRY(launch_finish_decode(plan, p->partials, tids, stream));
    if (!marks.mark(3)) return LORA_ERR_CUDA;
    p->n_calls += 1;
    return note_call(p, stream);
}

lora_status run_linear(lora_pool *p, const void *X, const void *W, const int32_t *ids, int T,
                       void *Y, cudaStream_t stream, bool with_lora)
{
    if (!p || !X || !W || !Y || (with_lora && !ids) || T < 0) return LORA_ERR_ARG;
    int path = p->path;
    if (path == LORA_PATH_DECODE && T > kDecodeMaxT) return LORA_ERR_ARG;
    if (path == LORA_PATH_AUTO && T > kDecodeMaxT && T <= kAutoDecodeMaxT) {
        // decode kernels over slices of kDecodeMaxT tokens: W streams once per slice, but
        // the adapters' A and B pages are read per token, never staged per segment (at
        // T = 512: 64 vs 167 us on tokens spread over 2000 adapters, 57 vs 75 us on
        // 8 contiguous adapters, against the prefill kernels)
        for (int t0 = 0; t0 < T; t0 += kDecodeMaxT) {
            const int n = T - t0 < kDecodeMaxT ? T - t0 : kDecodeMaxT;
            lora_status st = run_linear(p, static_cast<const uint16_t *>(X) + (size_t)t0 * p->d_in, W,
                                        with_lora ? ids + t0 : nullptr, n,
                                        static_cast<uint16_t *>(Y) + (size_t)t0 * p->d_out, stream, with_lora);
            if (st != LORA_OK) return st;
        }
        return LORA_OK;
    }
    if (path == LORA_PATH_AUTO) path = T <= kDecodeMaxT ? LORA_PATH_DECODE : LORA_PATH_PREFILL;
    if (T == 0) return LORA_OK;
    lora_status st = ensure_scratch(p, T);
    if (st != LORA_OK) return st;

    if ((st = order_after_changes(p, stream)) != LORA_OK) return st;
    const PoolDev pd = pool_view(p);
    const SegTables tabs = seg_tables(p);
    CallMarks marks{p, stream};
    if (!marks.begin()) return LORA_ERR_CUDA;
    auto mark = [&](int slot) { return marks.mark(slot); };
    const uint16_t *Xb = static_cast<const uint16_t *>(X);
    uint16_t *Yb = static_cast<uint16_t *>(Y);

    if (path == LORA_PATH_DECODE) {
        lora_pool *pools[1] = {p};
        st = run_decode(pools, 1, &X, &W, ids, T, &Y, stream, with_lora, marks);
        if (st != LORA_OK) return st;
    } else {
        // the segment tables; rows of the shrink output of tokens without an adapter zeroed
        uint64_t *tr = next_trace(p);
        if (with_lora)
            CUDA_TRY(launch_seg_build(ids, T, pd, tabs, p->d_err, p->Vhl, p->ldh, stream, trace_slot(tr, 0)));
        if (!mark(0)) return LORA_ERR_CUDA;
        const bool pair = p->pair_ok && (p->prefill_kernel == LORA_PREFILL_PAIR ||
                                         (p->prefill_kernel == LORA_PREFILL_AUTO && T > 128));
        CUtensorMap tmX, tmW, tmV, tmY;
        if (!tmap_for(p, &tmX, X, p->d_in, T, 64, 128) ||
            !tmap_for(p, &tmW, W, p->d_in, p->d_out, 64, pair ? 128 : 256) ||
            !tmap_for(p, &tmV, p->Vhl, p->ldh, T, 64, 128) || (pair && !tmap_for(p, &tmY, Y, p->d_out, T, 64, 32)))
            return LORA_ERR_ARG;
        if (with_lora) {
            CUDA_TRY(launch_shrink_small(Xb, T, pd, tabs, p->Vhl, p->ldh, p->num_sms, p->d_err, stream));
            CUDA_TRY(launch_shrink_tc(tmX, p->tmA, p->tmAw, Xb, T, pd, tabs, p->Vhl, p->ldh, p->num_sms,
                                      p->d_err, stream, trace_slot(tr, 1)));
        }
        if (!mark(1)) return LORA_ERR_CUDA;
        CUDA_TRY(launch_gemm_prefill(tmX, tmW, tmV, pair ? &p->tmB : nullptr, pair ? &tmY : nullptr, T,
                                     with_lora ? ids : nullptr,
                                     with_lora ? p->tile_info : nullptr, pd, p->Vhl, p->ldh, Yb,
                                     p->num_sms, p->d_err, stream, trace_slot(tr, 2)));
        if (!mark(2)) return LORA_ERR_CUDA;
    }
    p->n_calls += 1;
    return note_call(p, stream);
}

}  // namespace

// ===================================================================== C ABI

extern "C" {

int lora_abi_version(void) { return LORA_ABI_VERSION; }

const char *lora_status_string(lora_status s)
{
    switch (s) {
    case LORA_OK: return "ok";
    case LORA_ERR_ARG: return "invalid argument";
    case LORA_ERR_SHAPE: return "invalid shape";
    case LORA_ERR_SLOT_RANGE: return "slot out of range";
    case LORA_ERR_SLOT_OCCUPIED: return "slot already holds an adapter";
    case LORA_ERR_SLOT_EMPTY: return "slot is empty";
    case LORA_ERR_RANK: return "rank out of range";
    case LORA_ERR_BAD_ADAPTER_ID: return "a token id named no loaded adapter";
    case LORA_ERR_CUDA: return "CUDA error";
    case LORA_ERR_OOM: return "out of device memory";
    case LORA_ERR_TIMEOUT: return "a kernel wait timed out";
    case LORA_ERR_UNSUPPORTED: return "device is not compute capability 10.3";
    case LORA_ERR_IN_USE: return "a chain still lists this adapter";
    case LORA_ERR_RANGE: return "a checked kernel met an index out of range";
    }
    return "unknown status";
}

lora_status lora_pool_create(int max_adapters, int max_rank, int d_in, int d_out, lora_pool_t *out)
{
    if (!out) return LORA_ERR_ARG;
    *out = nullptr;
    if (max_adapters < 1 || max_adapters > LORA_MAX_ADAPTERS) return LORA_ERR_ARG;
    if (max_rank < 1 || max_rank > LORA_MAX_RANK) return LORA_ERR_RANK;
    if (!dims_ok(d_in) || !dims_ok(d_out)) return LORA_ERR_SHAPE;

    int dev = 0, major = 0, minor = 0, sms = 0;
    CUDA_TRY(cudaGetDevice(&dev));
    CUDA_TRY(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev));
    CUDA_TRY(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev));
    CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    if (major != 10 || minor != 3) return LORA_ERR_UNSUPPORTED;

    lora_pool *p = new (std::nothrow) lora_pool();
    if (!p) return LORA_ERR_OOM;
    p->device = dev;
    p->num_sms = sms;
    p->max_adapters = max_adapters;
    p->max_rank = max_rank;
    p->d_in = d_in;
    p->d_out = d_out;
    p->max_pages = (max_rank + kRankPage - 1) / kRankPage;
    // the zero page, room for max_adapters adapters at max_rank, and a reserve of two
    // adapters' pages so that a swap on a full pool can write pages no call still reads
    p->reserve_pages = 2 * p->max_pages;
    p->num_pages = max_adapters * p->max_pages + 1 + p->reserve_pages;
    // page ids, then one scale per page, and one more readable scale entry (the
    // tensor-core shrink reads the scale of the zero page that pads an odd count)
    p->slot_stride = ((slot_page_scale(p->max_pages, p->max_pages) + 1 + 3) / 4) * 4;
    p->ldv = ((p->max_pages * kRankPage + 15) / 16) * 16;
    p->ldh = 2 * (((p->max_pages * kRankPage + 31) / 32) * 32);
    p->h_slots.assign((size_t)max_adapters * p->slot_stride, 0);
    p->slot_copy_ev.assign(max_adapters, nullptr);
    p->chain_refs.assign(max_adapters, 0);
    p->free_pages.reserve(p->num_pages - 1);
    for (int pg = p->num_pages - 1; pg >= 1; --pg) p->free_pages.push_back(pg);

    const size_t a_bytes = (size_t)p->num_pages * kRankPage * d_in * 2;
    const size_t b_bytes = (size_t)p->num_pages * d_out * kRankPage * 2;
    lora_status st;
    if ((st = alloc_dev(p, (void **)&p->A_pages, a_bytes)) ||
        (st = alloc_dev(p, (void **)&p->B_pages, b_bytes)) ||
        (st = alloc_dev(p, (void **)&p->d_slots, sizeof(int32_t) * p->h_slots.size())) ||
        (st = alloc_dev(p, (void **)&p->d_err, 2 * sizeof(int))) ||
        (st = alloc_dev(p, (void **)&p->stage_A, (size_t)d_in * max_rank * 2)) ||
        (st = alloc_dev(p, (void **)&p->stage_B, (size_t)d_out * max_rank * 2)) ||
        (st = alloc_dev(p, (void **)&p->load_A, (size_t)d_in * max_rank * 2)) ||
        (st = alloc_dev(p, (void **)&p->load_B, (size_t)d_out * max_rank * 2)) ||
        (st = alloc_dev(p, (void **)&p->d_page_list, sizeof(int32_t) * p->max_pages)) ||
        (st = alloc_dev(p, (void **)&p->d_page_list_load, sizeof(int32_t) * p->max_pages))) {
        lora_pool_destroy(p);
        return st;
    }
    const size_t row_ints = (size_t)p->slot_stride + p->max_pages;
    if (cudaHostAlloc((void **)&p->stage_rows, sizeof(int32_t) * row_ints * (max_adapters + 1),
                      cudaHostAllocDefault) != cudaSuccess ||
        cudaHostAlloc((void **)&p->h_err, sizeof(int), cudaHostAllocDefault) != cudaSuccess) {
        cudaGetLastError();
        lora_pool_destroy(p);
        return LORA_ERR_OOM;
    }
    std::memset(p->stage_rows, 0, sizeof(int32_t) * row_ints * (max_adapters + 1));
    bool events_ok = cudaEventCreateWithFlags(&p->ev_call, cudaEventDisableTiming) == cudaSuccess &&
                     cudaEventCreateWithFlags(&p->ev_copy, cudaEventDisableTiming) == cudaSuccess &&
                     cudaEventCreateWithFlags(&p->ev_loaded, cudaEventDisableTiming) == cudaSuccess;
    for (int i = 0; events_ok && i < max_adapters; ++i)
        events_ok = cudaEventCreateWithFlags(&p->slot_copy_ev[i], cudaEventDisableTiming) == cudaSuccess;
    if (!events_ok ||
        cudaMemset(p->A_pages, 0, (size_t)kRankPage * d_in * 2) != cudaSuccess ||
        cudaMemset(p->B_pages, 0, (size_t)d_out * kRankPage * 2) != cudaSuccess ||
        cudaMemset(p->d_slots, 0, sizeof(int32_t) * p->h_slots.size()) != cudaSuccess ||
        cudaMemset(p->d_err, 0, 2 * sizeof(int)) != cudaSuccess ||
        cudaStreamCreateWithFlags(&p->copy_stream, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&p->load_stream, cudaStreamNonBlocking) != cudaSuccess ||
        // the kernels of loads, unloads and error reads are loaded now: a first launch
        // of a kernel not yet loaded (lazy module loading) can wait for the whole device
        ensure_smem_attr((const void *)pack_adapter_kernel, 0) != cudaSuccess ||
        ensure_smem_attr((const void *)read_clear_kernel, 0) != cudaSuccess ||
        !make_tmap_bf16_2d(&p->tmA, p->A_pages, d_in, (uint64_t)p->num_pages * kRankPage,
                           (uint64_t)d_in * 2, 64, kRankPage) ||
        !make_tmap_bf16_2d(&p->tmAw, p->A_pages, d_in, (uint64_t)p->num_pages * kRankPage,
                           (uint64_t)d_in * 2, 64,
                           (uint32_t)(((p->max_pages * kRankPage + 15) / 16) * 16)) ||
        cudaDeviceSynchronize() != cudaSuccess) {
        lora_pool_destroy(p);
        return LORA_ERR_CUDA;
    }
    // the CTA-pair prefill kernel reads the slice of a B page for its 128 columns (2 KB,
    // contiguous) with one TMA box: the arena viewed as rows of 64 values (8 columns of
    // 8 rank values), box 16 rows; the row coordinate is a 32-bit int
    const uint64_t b_rows = (uint64_t)p->num_pages * d_out / 8;
    p->pair_ok = b_rows + 32 < (1ull << 31) &&
                 make_tmap_bf16_2d(&p->tmB, p->B_pages, 64, b_rows, 128, 64, 16, false);
    *out = p;
    return LORA_OK;
}

lora_status lora_pool_destroy(lora_pool_t p)
{
    if (!p) return LORA_ERR_ARG;
    cudaDeviceSynchronize();
    destroy_host_tier(p);
    free_scratch(p);
    free_dev(p, p->hx, (size_t)p->cap_host_T * p->d_in * 2);
    free_dev(p, p->hy, (size_t)p->cap_host_T * p->d_out * 2);
    free_dev(p, p->hids, sizeof(int32_t) * (size_t)p->cap_host_T);
    free_dev(p, p->A_pages, 0);
    free_dev(p, p->B_pages, 0);
    free_dev(p, p->d_slots, 0);
    free_dev(p, p->d_err, 0);
    free_dev(p, p->stage_A, 0);
    free_dev(p, p->stage_B, 0);
    free_dev(p, p->load_A, 0);
    free_dev(p, p->wdq, 0);
    free_dev(p, p->load_B, 0);
    free_dev(p, p->d_page_list, 0);
    free_dev(p, p->d_page_list_load, 0);
    for (const lora_pool::FreedBatch &b : p->freed) cudaEventDestroy(b.ev);
    for (cudaEvent_t e : p->idle_events) cudaEventDestroy(e);
    if (p->copy_stream) cudaStreamDestroy(p->copy_stream);
    if (p->load_stream) cudaStreamDestroy(p->load_stream);
    for (auto &e : p->ev)
        if (e) cudaEventDestroy(e);
    for (cudaEvent_t e : p->slot_copy_ev)
        if (e) cudaEventDestroy(e);
    for (cudaEvent_t e : {p->ev_call, p->ev_copy, p->ev_loaded})
        if (e) cudaEventDestroy(e);
    if (p->stage_rows) cudaFreeHost(p->stage_rows);
    if (p->h_err) cudaFreeHost(p->h_err);
    delete p;
    return LORA_OK;
}

lora_status lora_pool_reserve(lora_pool_t p, int max_tokens)
{
    if (!p || max_tokens < 0) return LORA_ERR_ARG;
    return ensure_scratch(p, max_tokens);
}

lora_status lora_load_adapter(lora_pool_t p, int slot, const void *A, const void *B, int rank,
                              float alpha)
{
    if (!p || !A || !B) return LORA_ERR_ARG;
    if (slot < 0 || slot >= p->max_adapters) return LORA_ERR_SLOT_RANGE;
    if (rank < 1 || rank > p->max_rank) return LORA_ERR_RANK;
    int32_t *row = &p->h_slots[(size_t)slot * p->slot_stride];
    if (row[SLOT_RANK] != 0) return LORA_ERR_SLOT_OCCUPIED;
    const int npages = (rank + kRankPage - 1) / kRankPage;
    if (free_page_count(p) < npages) return LORA_ERR_OOM;

    // The caller's A and B into the pool's load buffers first, on a stream of their
    // own (not behind the pool's calls), so that the caller may free them on return;
    // the previous load's packing must have read those buffers.
    const size_t a_bytes = (size_t)p->d_in * rank * 2, b_bytes = (size_t)rank * p->d_out * 2;
    CUDA_TRY(cudaEventSynchronize(p->ev_loaded));
    int32_t *srow = nullptr;
    lora_status st = stage_row_ready(p, slot, &srow);
    if (st != LORA_OK) return st;
    int32_t *pages = srow + p->slot_stride;
    std::fill(srow, srow + p->slot_stride + p->max_pages, 0);
    bool fresh = false;
    take_pages(p, npages, pages, &fresh);
    // Pages that no enqueued call can read are written at once on the load stream,
    // behind the copies (the wait below covers both); pages freed by an unload whose
    // earlier calls may still be running are written on the copy stream after every
    // call enqueued on the pool so far. Either way the table row follows on the copy
    // stream, before every call enqueued from now on.
    cudaStream_t ps = fresh ? p->load_stream : p->copy_stream;
    int32_t *d_list = fresh ? p->d_page_list_load : p->d_page_list;
    if (cudaMemcpyAsync(p->load_A, A, a_bytes, cudaMemcpyDefault, p->load_stream) != cudaSuccess ||
        cudaMemcpyAsync(p->load_B, B, b_bytes, cudaMemcpyDefault, p->load_stream) != cudaSuccess ||
        (!fresh && cudaStreamSynchronize(p->load_stream) != cudaSuccess) ||
        cudaMemcpyAsync(d_list, pages, sizeof(int32_t) * npages, cudaMemcpyHostToDevice, ps) != cudaSuccess ||
        launch_pack_adapter(p->load_A, p->load_B, rank, d_list, npages, pool_view(p), p->A_pages,
                            p->B_pages, p->d_err, ps) != cudaSuccess ||
        cudaEventRecord(p->ev_loaded, ps) != cudaSuccess ||
        (fresh && cudaStreamSynchronize(p->load_stream) != cudaSuccess)) {
        cudaGetLastError();
        release_pages(p, pages, npages);  // back to the free list, after the calls so far
        return LORA_ERR_CUDA;
    }
    srow[SLOT_RANK] = rank;
    srow[SLOT_NPAGES] = npages;
    const float scale = alpha / (float)rank;
    std::memcpy(&srow[SLOT_SCALE], &scale, sizeof(float));
    for (int q = 0; q < npages; ++q) {
        srow[SLOT_PAGES + q] = pages[q];
        std::memcpy(&srow[slot_page_scale(p->max_pages, q)], &scale, sizeof(float));
    }
    if ((st = enqueue_row(p, slot, srow)) != LORA_OK) return st;
    std::copy(srow, srow + p->slot_stride, row);
    p->n_loads += 1;
    return LORA_OK;
}

lora_status lora_unload_adapter(lora_pool_t p, int slot)
{
    if (!p) return LORA_ERR_ARG;
    if (slot < 0 || slot >= p->max_adapters) return LORA_ERR_SLOT_RANGE;
    int32_t *row = &p->h_slots[(size_t)slot * p->slot_stride];
    if (row[SLOT_RANK] == 0) return LORA_ERR_SLOT_EMPTY;
    if (p->chain_refs[slot] > 0) return LORA_ERR_IN_USE;  // a chain still lists it
    if (slot_is_held(p, slot)) return LORA_ERR_IN_USE;    // acquired from the host tier
    // the empty row goes in on the copy stream, after the calls enqueued so far; the
    // pages are free once those calls have run
    int32_t *zero = nullptr;
    lora_status st = stage_row_ready(p, p->max_adapters, &zero);
    if (st != LORA_OK) return st;
    if ((st = enqueue_row(p, slot, zero)) != LORA_OK) return st;
    const int npages = row[SLOT_NPAGES];
    if (row[SLOT_MEMBERS] > 0) {
        // a chain owns no pages: release its members
        for (int m : p->chain_members[slot]) p->chain_refs[m] -= 1;
        p->chain_members.erase(slot);
    } else if ((st = release_pages(p, &row[SLOT_PAGES], npages)) != LORA_OK) {
        return st;
    }
    std::fill(row, row + p->slot_stride, 0);
    forget_cached_slot(p, slot);
    p->n_unloads += 1;
    return LORA_OK;
}

lora_status lora_define_chain(lora_pool_t p, int chain_slot, const int *member_slots, int n)
{
    if (!p || !member_slots || n < 1) return LORA_ERR_ARG;
    if (chain_slot < 0 || chain_slot >= p->max_adapters) return LORA_ERR_SLOT_RANGE;
    int32_t *row = &p->h_slots[(size_t)chain_slot * p->slot_stride];
    if (row[SLOT_RANK] != 0) return LORA_ERR_SLOT_OCCUPIED;
    std::vector<int32_t> new_row(p->slot_stride, 0);
    int rank = 0, npages = 0;
    for (int e = 0; e < n; ++e) {
        const int m = member_slots[e];
        if (m < 0 || m >= p->max_adapters) return LORA_ERR_SLOT_RANGE;
        const int32_t *mrow = &p->h_slots[(size_t)m * p->slot_stride];
        if (mrow[SLOT_RANK] == 0) return LORA_ERR_SLOT_EMPTY;
        if (mrow[SLOT_MEMBERS] > 0 || m == chain_slot) return LORA_ERR_ARG;  // members are adapters
        for (int k = 0; k < e; ++k)
            if (member_slots[k] == m) return LORA_ERR_ARG;  // each member once
        const int mp = mrow[SLOT_NPAGES];
        if (npages + mp > p->max_pages) return LORA_ERR_RANK;  // the chain's pages fit one row
        for (int q = 0; q < mp; ++q) {
            new_row[SLOT_PAGES + npages + q] = mrow[SLOT_PAGES + q];
            new_row[slot_page_scale(p->max_pages, npages + q)] =
                mrow[slot_page_scale(p->max_pages, q)];
        }
        npages += mp;
        rank += mrow[SLOT_RANK];
    }
    new_row[SLOT_RANK] = rank;
    new_row[SLOT_NPAGES] = npages;
    new_row[SLOT_SCALE] = p->h_slots[(size_t)member_slots[0] * p->slot_stride + SLOT_SCALE];
    new_row[SLOT_MEMBERS] = n;
    // the row goes in on the copy stream: calls enqueued before see the slot empty
    int32_t *srow = nullptr;
    lora_status st = stage_row_ready(p, chain_slot, &srow);
    if (st != LORA_OK) return st;
    std::copy(new_row.begin(), new_row.end(), srow);
    if ((st = enqueue_row(p, chain_slot, srow)) != LORA_OK) return st;
    std::copy(new_row.begin(), new_row.end(), row);
    std::vector<int> &members = p->chain_members[chain_slot];
    members.assign(member_slots, member_slots + n);
    for (int m : members) p->chain_refs[m] += 1;
    return LORA_OK;
}

lora_status lora_linear(lora_pool_t p, const void *X, const void *W_base,
                        const int32_t *token_adapter_ids, int T, void *Y, lora_stream_t stream)
{
    return run_linear(p, X, W_base, token_adapter_ids, T, Y, (cudaStream_t)stream, true);
}

lora_status lora_base_linear(lora_pool_t p, const void *X, const void *W_base, int T, void *Y,
                             lora_stream_t stream)
{
    return run_linear(p, X, W_base, nullptr, T, Y, (cudaStream_t)stream, false);
}

lora_status lora_linear_q4(lora_pool_t p, const void *X, const void *Wq, const void *scales,
                           const void *zeros, const int32_t *token_adapter_ids, int T, void *Y,
                           lora_stream_t stream)
{
    return run_linear_q4(p, X, Wq, scales, zeros, token_adapter_ids, T, Y, (cudaStream_t)stream, true);
}

lora_status lora_base_linear_q4(lora_pool_t p, const void *X, const void *Wq, const void *scales,
                                const void *zeros, int T, void *Y, lora_stream_t stream)
{
    return run_linear_q4(p, X, Wq, scales, zeros, nullptr, T, Y, (cudaStream_t)stream, false);
}

lora_status lora_dequant_q4(const void *Wq, const void *scales, const void *zeros, int d_out, int d_in,
                            void *W, lora_stream_t stream)
{
    if (!Wq || !scales || !zeros || !W) return LORA_ERR_ARG;
    if (!dims_ok(d_in) || !dims_ok(d_out) || d_in % kQ4Group != 0) return LORA_ERR_SHAPE;
    if (((uintptr_t)Wq | (uintptr_t)W) & 15) return LORA_ERR_ARG;  // 4- and 16-byte accesses
    CUDA_TRY(launch_dequant_q4(static_cast<const uint8_t *>(Wq), static_cast<const uint16_t *>(scales),
                               static_cast<const uint8_t *>(zeros), d_out, d_in, static_cast<uint16_t *>(W),
                               (cudaStream_t)stream));
    return LORA_OK;
}

lora_status lora_linear_grouped(int n, const lora_pool_t *pools, const void *const *X,
                                const void *const *W_base, const int32_t *token_adapter_ids, int T,
                                void *const *Y, lora_stream_t stream)
{
    if (n < 1 || n > LORA_MAX_GROUP || !pools || !X || !W_base || !token_adapter_ids || !Y || T < 0)
        return LORA_ERR_ARG;
    for (int m = 0; m < n; ++m) {
        if (!pools[m] || !X[m] || !W_base[m] || !Y[m]) return LORA_ERR_ARG;
        if (pools[m]->device != pools[0]->device) return LORA_ERR_ARG;
        for (int k = 0; k < m; ++k)
            if (pools[k] == pools[m]) return LORA_ERR_ARG;  // each problem uses its pool's scratch
    }
    if (T == 0) return LORA_OK;
    cudaStream_t s = (cudaStream_t)stream;
    int path = pools[0]->path;
    if (path == LORA_PATH_AUTO) path = T <= kDecodeMaxT ? LORA_PATH_DECODE : LORA_PATH_PREFILL;
    if (path == LORA_PATH_DECODE && T > kDecodeMaxT) return LORA_ERR_ARG;
    if (path == LORA_PATH_PREFILL) {
        // prefill-sized batches: the layers one after another, each on its own path
        for (int m = 0; m < n; ++m) {
            lora_status st = run_linear(pools[m], X[m], W_base[m], token_adapter_ids, T, Y[m], s, true);
            if (st != LORA_OK) return st;
        }
        return LORA_OK;
    }
    for (int m = 0; m < n; ++m) {
        lora_status st = ensure_scratch(pools[m], T);
        if (st == LORA_OK) st = order_after_changes(pools[m], s);
        if (st != LORA_OK) return st;
    }
    CallMarks marks{pools[0], s};
    if (!marks.begin()) return LORA_ERR_CUDA;
    lora_status st = run_decode(pools, n, X, W_base, token_adapter_ids, T, Y, s, true, marks);
    if (st != LORA_OK) return st;
    for (int m = 0; m < n; ++m) {
        pools[m]->n_calls += 1;
        st = note_call(pools[m], s);
        if (st != LORA_OK) return st;
    }
    return LORA_OK;
}

lora_status lora_linear_host(lora_pool_t p, const void *X_host, const void *W_base,
                             const int32_t *ids_host, int T, void *Y_host, lora_stream_t stream)
{
    if (!p || !X_host || !W_base || !ids_host || !Y_host || T < 0) return LORA_ERR_ARG;
    if (T == 0) return LORA_OK;
    if (T > p->cap_host_T) {
        CUDA_TRY(cudaDeviceSynchronize());
        free_dev(p, p->hx, (size_t)p->cap_host_T * p->d_in * 2);
        free_dev(p, p->hy, (size_t)p->cap_host_T * p->d_out * 2);
        free_dev(p, p->hids, sizeof(int32_t) * (size_t)p->cap_host_T);
        p->hx = p->hy = nullptr;
        p->hids = nullptr;
        p->cap_host_T = 0;
        lora_status st;
        if ((st = alloc_dev(p, (void **)&p->hx, (size_t)T * p->d_in * 2)) ||
            (st = alloc_dev(p, (void **)&p->hy, (size_t)T * p->d_out * 2)) ||
            (st = alloc_dev(p, (void **)&p->hids, sizeof(int32_t) * (size_t)T)))
            return st;
        p->cap_host_T = T;
    }
    cudaStream_t s = (cudaStream_t)stream;
    CUDA_TRY(cudaMemcpyAsync(p->hx, X_host, (size_t)T * p->d_in * 2, cudaMemcpyHostToDevice, s));
    CUDA_TRY(cudaMemcpyAsync(p->hids, ids_host, sizeof(int32_t) * (size_t)T, cudaMemcpyHostToDevice, s));
    lora_status st = run_linear(p, p->hx, W_base, p->hids, T, p->hy, s, true);
    if (st != LORA_OK) return st;
    CUDA_TRY(cudaMemcpyAsync(Y_host, p->hy, (size_t)T * p->d_out * 2, cudaMemcpyDeviceToHost, s));
    CUDA_TRY(cudaStreamSynchronize(s));
    return LORA_OK;
}

lora_status lora_decode_plan_info(int n, int T, const int *d_in, const int *d_out,
                                  const int *max_pages, int num_sms, int64_t *out)
{
    if (!d_in || !d_out || !max_pages || !out) return LORA_ERR_ARG;
    for (int m = 0; m < n && m < kMaxGroup; ++m)
        if (!dims_ok(d_in[m]) || !dims_ok(d_out[m]) || max_pages[m] < 0) return LORA_ERR_SHAPE;
    DecodePlan p;
    if (!plan_decode(n, T, d_in, d_out, max_pages, num_sms, &p)) return LORA_ERR_ARG;
    const int64_t v[LORA_PLAN_INFO_COUNT] = {p.U, p.G, p.grid, p.max_seg, p.n_acc, p.stages,
                                             (int64_t)p.tmem_cols, (int64_t)p.smem_bytes, p.pairs,
                                             p.col_blocks, p.tight ? 1 : 0, p.ntok,
                                             (int64_t)decode_partials_floats(p),
                                             p.prefetch_a ? 1 : 0};
    for (int i = 0; i < LORA_PLAN_INFO_COUNT; ++i) out[i] = v[i];
    return LORA_OK;
}

lora_status lora_pool_selftest_wait(lora_pool_t p, int limit_us, lora_stream_t stream)
{
    if (!p || limit_us < 1 || limit_us > 2000000) return LORA_ERR_ARG;
    wait_selftest_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(p->d_err, (uint64_t)limit_us * 1000ull);
    CUDA_TRY(cudaGetLastError());
    return LORA_OK;
}

lora_status lora_test_delayed_copy(const int32_t *src, int32_t *dst, int n, int delay_us, lora_stream_t stream)
{
    if (!src || !dst || n < 0 || delay_us < 1 || delay_us > 100000) return LORA_ERR_ARG;
    delayed_copy_kernel<<<1, 256, 0, (cudaStream_t)stream>>>(src, dst, n, (uint64_t)delay_us * 1000ull);
    CUDA_TRY(cudaGetLastError());
    return LORA_OK;
}

lora_status lora_pool_check_errors(lora_pool_t p)
{
    if (!p) return LORA_ERR_ARG;
    // on the copy stream, which follows every call enqueued on the pool: the word is
    // read and cleared in one atomic step (a kernel still running on another stream
    // cannot set a bit between the read and the clear and have it lost)
    cudaStream_t s = p->copy_stream;
    read_clear_kernel<<<1, 1, 0, s>>>(p->d_err);
    if (cudaGetLastError() != cudaSuccess ||
        cudaMemcpyAsync(p->h_err, p->d_err + 1, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return LORA_ERR_CUDA;
    const int word = *p->h_err;
    if (word & kErrBadIdBit) return LORA_ERR_BAD_ADAPTER_ID;
    if (word & kErrTimeoutBit) return LORA_ERR_TIMEOUT;
    if (word & kErrRangeBit) return LORA_ERR_RANGE;
    return LORA_OK;
}

lora_status lora_build_segments(lora_pool_t p, const int32_t *ids, int T, int32_t *order,
                                int32_t *n_base, int32_t *num_seg, int32_t *seg_start,
                                int32_t *seg_slot, lora_stream_t stream)
{
    if (!p || !ids || !order || !n_base || !num_seg || !seg_start || !seg_slot || T < 0)
        return LORA_ERR_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    if (T == 0) {
        CUDA_TRY(cudaMemsetAsync(n_base, 0, sizeof(int32_t), s));
        CUDA_TRY(cudaMemsetAsync(num_seg, 0, sizeof(int32_t), s));
        CUDA_TRY(cudaMemsetAsync(seg_start, 0, sizeof(int32_t), s));
        return LORA_OK;
    }
    lora_status st = ensure_scratch(p, T);
    if (st == LORA_OK) st = order_after_changes(p, s);
    if (st != LORA_OK) return st;
    const SegTables tabs = seg_tables(p);
    CUDA_TRY(launch_seg_build(ids, T, pool_view(p), tabs, p->d_err, nullptr, 0, s));
    const size_t se = seg_entries(p, T);
    CUDA_TRY(cudaMemcpyAsync(order, p->order, sizeof(int32_t) * T, cudaMemcpyDeviceToDevice, s));
    CUDA_TRY(cudaMemcpyAsync(n_base, p->hdr + HDR_NBASE, sizeof(int32_t), cudaMemcpyDeviceToDevice, s));
    CUDA_TRY(cudaMemcpyAsync(num_seg, p->hdr + HDR_NUMSEG, sizeof(int32_t), cudaMemcpyDeviceToDevice, s));
    CUDA_TRY(cudaMemcpyAsync(seg_start, p->seg_start, sizeof(int32_t) * se, cudaMemcpyDeviceToDevice, s));
    CUDA_TRY(cudaMemcpyAsync(seg_slot, p->seg_slot, sizeof(int32_t) * (se - 1), cudaMemcpyDeviceToDevice, s));
    return note_call(p, s);
}

lora_status lora_pool_stats(lora_pool_t p, int64_t *out)
{
    if (!p || !out) return LORA_ERR_ARG;
    int64_t loaded = 0;
    for (int i = 0; i < p->max_adapters; ++i)
        if (p->h_slots[(size_t)i * p->slot_stride + SLOT_RANK] != 0) ++loaded;
    out[0] = loaded;
    // pages for loads, without the zero page and the reserve (loaded adapters never
    // hold more than max_adapters * max_pages pages, so the free count covers it)
    out[1] = std::max<int64_t>(0, (int64_t)free_page_count(p) - p->reserve_pages);
    out[2] = (int64_t)p->num_pages - 1 - p->reserve_pages;
    out[3] = p->n_loads;
    out[4] = p->n_unloads;
    out[5] = p->n_calls;
    out[6] = (int64_t)p->bytes_held;
    return LORA_OK;
}

lora_status lora_pool_enable_timing(lora_pool_t p, int enable)
{
    if (!p) return LORA_ERR_ARG;
    if (enable && !p->ev[0]) {
        for (auto &e : p->ev) CUDA_TRY(cudaEventCreate(&e));
    }
    p->timing = enable != 0;
    return LORA_OK;
}

lora_status lora_pool_kernel_times(lora_pool_t p, float *ms)
{
    if (!p || !ms) return LORA_ERR_ARG;
    for (int k = 0; k < LORA_KERNEL_SLOTS; ++k) ms[k] = 0.f;
    if (!p->ev[0]) return LORA_OK;
    CUDA_TRY(cudaEventSynchronize(p->ev[p->ev_last]));
    // slots are contiguous in launch order; an unused slot has no event of its own
    int prev = 0;
    for (int k = 0; k < LORA_KERNEL_SLOTS; ++k) {
        if (!p->ev_used[k]) continue;
        float t = 0.f;
        CUDA_TRY(cudaEventElapsedTime(&t, p->ev[prev], p->ev[k + 1]));
        ms[k] = t;
        prev = k + 1;
    }
    return LORA_OK;
}

lora_status lora_pool_set_trace(lora_pool_t p, uint64_t *buf, int n_calls)
{
    if (!p || (buf && n_calls < 1)) return LORA_ERR_ARG;
    p->trace = buf;
    p->trace_calls = buf ? n_calls : 0;
    p->trace_k = 0;
    return LORA_OK;
}

lora_status lora_pool_set_path(lora_pool_t p, int path)
{
    if (!p || path < LORA_PATH_AUTO || path > LORA_PATH_PREFILL) return LORA_ERR_ARG;
    p->path = path;
    return LORA_OK;
}

lora_status lora_pool_set_prefill_kernel(lora_pool_t p, int kernel)
{
    if (!p || kernel < LORA_PREFILL_AUTO || kernel > LORA_PREFILL_PAIR) return LORA_ERR_ARG;
    if (kernel == LORA_PREFILL_PAIR && !p->pair_ok) return LORA_ERR_UNSUPPORTED;
    p->prefill_kernel = kernel;
    return LORA_OK;
}

}  // extern "C"

// ============================================================== helpers

namespace lora {

cudaError_t launch_pack_adapter(const uint16_t *A, const uint16_t *B, int rank, const int32_t *pages,
                                int npages, const PoolDev &pool, uint16_t *A_pages,
                                uint16_t *B_pages, int *err, cudaStream_t stream)
{
    cudaError_t e = ensure_smem_attr((const void *)pack_adapter_kernel, 0);
    if (e != cudaSuccess) return e;
    const size_t total = (size_t)npages * kRankPage * (pool.d_in + pool.d_out);
    int grid = (int)std::min<size_t>((total + 255) / 256, 4096);
    pack_adapter_kernel<<<grid, 256, 0, stream>>>(A, B, rank, pages, npages, pool.d_in, pool.d_out,
                                                  A_pages, B_pages, pool.num_pages, err);
    return cudaGetLastError();
}

cudaError_t ensure_smem_attr(const void *kernel, size_t bytes)
{
    struct Entry {
        const void *kernel;
        int device;
        size_t bytes;
    };
    static std::mutex mu;
    static std::vector<Entry> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    for (Entry &x : done)
        if (x.kernel == kernel && x.device == dev) {
            if (x.bytes >= bytes) return cudaSuccess;
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
            if (e == cudaSuccess) x.bytes = bytes;
            return e;
        }
    // every kernel of the library asks for the largest shared-memory carveout, so an SM
    // never has to drain and reconfigure between two of them and kernels launched with
    // programmatic serialization can be resident beside the GEMM kernels
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess && bytes > 0)
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess) done.push_back({kernel, dev, bytes});
    return e;
}

static PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return encode;
}

bool make_tmap_u8_2d(CUtensorMap *map, const void *base, uint64_t inner, uint64_t rows,
                     uint64_t row_pitch_bytes, uint32_t box_inner, uint32_t box_rows)
{
    PFN_cuTensorMapEncodeTiled_v12000 encode = tmap_encoder();
    if (!encode || rows == 0) return false;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {row_pitch_bytes};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tmap_bf16_2d(CUtensorMap *map, const void *base, uint64_t inner, uint64_t rows,
                       uint64_t row_pitch_bytes, uint32_t box_inner, uint32_t box_rows, bool swizzle128)
{
    PFN_cuTensorMapEncodeTiled_v12000 encode = tmap_encoder();
    if (!encode || rows == 0) return false;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {row_pitch_bytes};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims,
                              strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace lora
