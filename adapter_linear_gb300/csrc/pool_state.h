// pool_state.h -- the host-side state of a lora_pool (private to the library):
// the paged arenas, the slot table and its host mirror, per-call scratch, the
// measurement hook and the host-tier adapter cache. pool.cu implements the pool
// and the layer calls, cache.cu the host tier.
#pragma once

#include <climits>
#include <deque>
#include <map>
#include <unordered_map>
#include <vector>

#include <cudaTypedefs.h>

#include "../../include/lora_linear.h"
#include "internal.h"

#define CUDA_TRY(expr)                                  \
    do {                                                \
        cudaError_t e_ = (expr);                        \
        if (e_ != cudaSuccess) return LORA_ERR_CUDA;    \
    } while (0)

struct TmapEntry {
    const void *base = nullptr;
    uint64_t inner = 0, rows = 0;
    uint32_t box_inner = 0, box_rows = 0;
    CUtensorMap map;
};

// One adapter of the host tier: pool-owned pinned copies of A and B.
struct HostAdapter {
    void *A = nullptr, *B = nullptr;  // pinned, the lora_load_adapter layouts
    int rank = 0;
    float alpha = 0.f;
    int slot = -1;                    // the GPU slot it occupies, or -1
};

constexpr int64_t kNoKey = INT64_MIN;

struct lora_pool {
    int device = 0, num_sms = 0;
    int max_adapters = 0, max_rank = 0, d_in = 0, d_out = 0;
    int max_pages = 0;   // pages per adapter at max_rank
    int num_pages = 0;   // arena pages, page 0 = zero page
    int reserve_pages = 0;  // arena pages beyond max_adapters * max_pages (see free_pages)
    int slot_stride = 0;
    int ldv = 0;         // fp32 row stride of the decode path's low-rank intermediate
    int ldh = 0;         // bf16 row stride of the prefill path's hi/lo intermediate
    uint16_t *A_pages = nullptr, *B_pages = nullptr;
    int32_t *d_slots = nullptr;
    std::vector<int32_t> h_slots;
    // Free pages that no enqueued layer call can read (stack; back() is taken first).
    // Pages an unload or eviction gives back may still be read by the calls enqueued
    // before it: they wait in `freed`, a batch per change with an event recorded on the
    // copy stream after it, and join free_pages once that event has completed. A load
    // that finds enough free pages writes them at once, beside the running calls; the
    // reserve pages let a swap on a full pool do so too.
    std::vector<int32_t> free_pages;
    struct FreedBatch {
        cudaEvent_t ev;
        std::vector<int32_t> pages;
    };
    std::deque<FreedBatch> freed;
    std::vector<cudaEvent_t> idle_events;  // recorded-and-completed batch events, for reuse
    std::vector<int32_t> chain_refs;  // per slot: chains that list it as a member
    std::map<int, std::vector<int>> chain_members;  // chain slot -> member slots
    int *d_err = nullptr;             // [0] the error word, [1] its value at the last read
    int *h_err = nullptr;             // pinned copy of d_err[1]
    uint16_t *stage_A = nullptr, *stage_B = nullptr;  // swap-ins of the host tier
    uint16_t *load_A = nullptr, *load_B = nullptr;    // lora_load_adapter's copy of A, B
    uint16_t *wdq = nullptr;  // a 4-bit base dequantised to bf16 for the prefill path (first use)
    int32_t *d_page_list = nullptr;       // page list of a packing on the copy stream
    int32_t *d_page_list_load = nullptr;  // ... on the load stream
    // Changes of pages and table rows (loads, unloads, chains, swap-ins) run on the
    // copy stream, which waits for every layer call enqueued on the pool before them;
    // layer calls enqueued after a change wait for the copy stream (ev_copy).
    cudaStream_t copy_stream = nullptr;
    cudaStream_t load_stream = nullptr;   // caller's A, B -> load_A, load_B
    cudaEvent_t ev_loaded = nullptr;      // the last packing of load_A, load_B
    uint64_t copy_epoch = 0;              // changes enqueued on the copy stream so far
    uint64_t waited_epoch = 0;            // ... that waited_stream was last made to wait for
    cudaStream_t waited_stream = nullptr;
    CUtensorMap tmA;   // A arena [num_pages*8 rows x d_in], box 8 x 64
    CUtensorMap tmAw;  // the same, box round16(8 * max_pages) x 64
    CUtensorMap tmB;   // B arena as [num_pages*d_out/8 rows x 64], box 16 x 64, no swizzle
    bool pair_ok = false;  // tmB exists (rows < 2^31): the CTA-pair prefill kernel can run

    // per-call scratch, sized for cap_T tokens
    int cap_T = 0;
    int32_t *order = nullptr, *hdr = nullptr, *seg_start = nullptr, *seg_slot = nullptr,
            *seg_ublk = nullptr, *tile_info = nullptr;
    int32_t *seg_keys = nullptr, *seg_chist = nullptr, *seg_ticket = nullptr;  // multi-CTA builder
    float *V = nullptr;
    uint16_t *Vhl = nullptr;
    float *partials = nullptr;
    size_t partials_floats = 0;
    // device staging of lora_linear_host
    int cap_host_T = 0;
    uint16_t *hx = nullptr, *hy = nullptr;
    int32_t *hids = nullptr;

    TmapEntry tmaps[8];
    int tmap_next = 0;

    int path = LORA_PATH_AUTO;
    int prefill_kernel = LORA_PREFILL_AUTO;
    bool timing = false;
    cudaEvent_t ev[LORA_KERNEL_SLOTS + 1] = {};
    bool ev_used[LORA_KERNEL_SLOTS] = {};
    int ev_last = 0;  // index of the last event the last timed call recorded
    // span trace (lora_pool_set_trace): call k of the pool since it was set writes
    // its kernels' (first entry, last exit) into trace[(k % trace_calls)][slot][2]
    uint64_t *trace = nullptr;
    int trace_calls = 0;
    int64_t trace_k = 0;
    int64_t n_loads = 0, n_unloads = 0, n_calls = 0;
    size_t bytes_held = 0;

    // marks each layer call enqueued directly on a stream (not inside a graph
    // capture) for the copy stream to wait on: every later change starts after it
    cudaEvent_t ev_call = nullptr;

    // host tier (cache.cu): key -> host copy; per slot the cached key it holds
    // (kNoKey: a manual or empty slot), acquisitions outstanding and last use.
    // Per slot (all slots, manual ones included): the copy that last wrote its
    // table row from its pinned staging row (reused only after that copy has run)
    std::unordered_map<int64_t, HostAdapter> host_tier;
    std::vector<int64_t> slot_key;
    std::vector<int32_t> slot_pins;
    std::vector<uint64_t> slot_tick;
    std::vector<cudaEvent_t> slot_copy_ev;
    int32_t *stage_rows = nullptr;  // pinned [max_adapters + 1][slot_stride + max_pages];
                                    // the last row stays all zero (empty slot)
    cudaEvent_t ev_copy = nullptr;  // the last change enqueued on copy_stream
    uint64_t tick = 0;
    int64_t cache_hits = 0, cache_misses = 0, cache_evictions = 0;
};

namespace lora {
lora_status alloc_dev(lora_pool *p, void **ptr, size_t bytes);
void free_dev(lora_pool *p, void *ptr, size_t bytes);
PoolDev pool_view(const lora_pool *p);
// Before a layer call on `stream`: order it after the page and table changes
// enqueued on the copy stream so far.
lora_status order_after_changes(lora_pool *p, cudaStream_t stream);
// After a layer call on `stream`: later changes on the copy stream wait for it.
lora_status note_call(lora_pool *p, cudaStream_t stream);
// The pinned staging row of `slot` (slot == max_adapters: the all-zero row), once
// the copy that last read it has run.
lora_status stage_row_ready(lora_pool *p, int slot, int32_t **row);
// Enqueue the copy of a staging row into the device table row of `slot` on the
// copy stream; later layer calls are ordered after it.
lora_status enqueue_row(lora_pool *p, int slot, const int32_t *row);
// Pages given back by an unload or eviction whose table change was just enqueued on
// the copy stream: free once the calls enqueued before it have run.
lora_status release_pages(lora_pool *p, const int32_t *pages, int n);
// Free pages, those still waiting for earlier calls included.
int free_page_count(const lora_pool *p);
// Take n free pages into out[] (the caller checked free_page_count). *fresh: every
// page taken is free of enqueued readers, so it may be written before the calls
// already enqueued have run; otherwise it must be written on the copy stream.
void take_pages(lora_pool *p, int n, int32_t *out, bool *fresh);
// Free the host tier's pinned memory and events (pool destruction).
void destroy_host_tier(lora_pool *p);
// A slot the host tier holds for an outstanding acquisition?
bool slot_is_held(const lora_pool *p, int slot);
// A cached slot emptied through lora_unload_adapter: drop it from the tier.
void forget_cached_slot(lora_pool *p, int slot);
}  // namespace lora
