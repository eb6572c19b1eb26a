// cache.cu -- the host tier of the adapter pool: more adapters than the GPU
// slots hold, kept in pinned host memory and swapped into the pool on demand.
//
// The pages describe this tier: the adapters stay on the host (or disk) and the
// GPU pool caches the active ones, loading a missing adapter when a request
// names it and swapping out the least recently used one when the pool is full
// (icman.com.cn Multi-LoRA article, sections 2.1 and 2.2; the vLLM tutorial's
// "max-loras vs max-cpu-loras" section: a GPU-resident set backed by a larger
// CPU-resident set). The same article's section 4.2 blames cold adapter loads
// for latency spikes; here a swap-in never blocks the host or the caller's
// stream beyond the copy itself:
//  * every layer call on the pool makes the pool's copy stream wait for it, and
//    a swap-in is enqueued on that stream: it starts after the calls enqueued
//    before it (which may still read the evicted pages or the slot's table
//    row), copies A and B from pinned memory, packs them into pages and writes
//    the slot's table row;
//  * lora_acquire makes the caller's stream wait for the last swap-in, so the
//    next layer call on that stream sees the adapter;
//  * eviction picks the cached slot used least recently among those with no
//    acquisition outstanding and no chain listing them; manually loaded slots
//    are never evicted.
#include <algorithm>
#include <cstring>

#include "pool_state.h"

using namespace lora;

namespace {

lora_status ensure_tier(lora_pool *p)
{
    if (!p->slot_key.empty()) return LORA_OK;
    p->slot_key.assign(p->max_adapters, kNoKey);
    p->slot_pins.assign(p->max_adapters, 0);
    p->slot_tick.assign(p->max_adapters, 0);
    return LORA_OK;
}

// Take cached slot s out of the GPU: its table row is cleared and its pages are
// freed (asynchronously, after the calls already enqueued).
lora_status evict(lora_pool *p, int s)
{
    int32_t *row = &p->h_slots[(size_t)s * p->slot_stride];
    int32_t *zero = nullptr;
    lora_status st = stage_row_ready(p, p->max_adapters, &zero);
    if (st != LORA_OK) return st;
    if ((st = enqueue_row(p, s, zero)) != LORA_OK) return st;
    if ((st = release_pages(p, &row[SLOT_PAGES], row[SLOT_NPAGES])) != LORA_OK) return st;
    std::fill(row, row + p->slot_stride, 0);
    p->host_tier[p->slot_key[s]].slot = -1;
    p->slot_key[s] = kNoKey;
    p->slot_tick[s] = 0;
    p->n_unloads += 1;
    p->cache_evictions += 1;
    return LORA_OK;
}

// The empty slot the tier takes (searched from the top, away from the low slots
// that manual loads usually use), or -1.
int empty_slot(const lora_pool *p)
{
    for (int s = p->max_adapters - 1; s >= 0; --s)
        if (p->h_slots[(size_t)s * p->slot_stride + SLOT_RANK] == 0 && p->slot_key[s] == kNoKey)
            return s;
    return -1;
}

// The cached slot used least recently with nothing holding it, or -1.
int lru_victim(const lora_pool *p)
{
    int best = -1;
    for (int s = 0; s < p->max_adapters; ++s) {
        if (p->slot_key[s] == kNoKey || p->slot_pins[s] > 0 || p->chain_refs[s] > 0) continue;
        if (best < 0 || p->slot_tick[s] < p->slot_tick[best]) best = s;
    }
    return best;
}

// Make `key` resident: free a slot and pages (evicting as needed) and enqueue the
// copy of its pinned A and B into them.
lora_status swap_in(lora_pool *p, int64_t key, HostAdapter &h)
{
    const int npages = (h.rank + kRankPage - 1) / kRankPage;
    int slot = empty_slot(p);
    while (slot < 0 || free_page_count(p) < npages) {
        const int victim = lru_victim(p);
        if (victim < 0) return LORA_ERR_OOM;  // everything left is held
        lora_status st = evict(p, victim);
        if (st != LORA_OK) return st;
        if (slot < 0) slot = empty_slot(p);
    }
    // the slot's staging row may still be read by its previous table copy
    int32_t *row = nullptr;
    lora_status st = stage_row_ready(p, slot, &row);
    if (st != LORA_OK) return st;
    int32_t *pages = row + p->slot_stride;
    std::fill(row, row + p->slot_stride + p->max_pages, 0);
    bool fresh = false;  // written on the copy stream, after the calls, in any case
    take_pages(p, npages, pages, &fresh);
    const float scale = h.alpha / (float)h.rank;
    row[SLOT_RANK] = h.rank;
    row[SLOT_NPAGES] = npages;
    std::memcpy(&row[SLOT_SCALE], &scale, sizeof(float));
    for (int q = 0; q < npages; ++q) {
        row[SLOT_PAGES + q] = pages[q];
        std::memcpy(&row[slot_page_scale(p->max_pages, q)], &scale, sizeof(float));
    }

    cudaStream_t s = p->copy_stream;
    const size_t a_bytes = (size_t)p->d_in * h.rank * 2, b_bytes = (size_t)h.rank * p->d_out * 2;
    CUDA_TRY(cudaMemcpyAsync(p->stage_A, h.A, a_bytes, cudaMemcpyHostToDevice, s));
    CUDA_TRY(cudaMemcpyAsync(p->stage_B, h.B, b_bytes, cudaMemcpyHostToDevice, s));
    CUDA_TRY(cudaMemcpyAsync(p->d_page_list, pages, sizeof(int32_t) * npages,
                             cudaMemcpyHostToDevice, s));
    CUDA_TRY(launch_pack_adapter(p->stage_A, p->stage_B, h.rank, p->d_page_list, npages,
                                 pool_view(p), p->A_pages, p->B_pages, p->d_err, s));
    if ((st = enqueue_row(p, slot, row)) != LORA_OK) return st;

    std::copy(row, row + p->slot_stride, &p->h_slots[(size_t)slot * p->slot_stride]);
    p->slot_key[slot] = key;
    h.slot = slot;
    p->n_loads += 1;
    return LORA_OK;
}

}  // namespace

namespace lora {

// Called when a cached slot is unloaded through lora_unload_adapter.
void forget_cached_slot(lora_pool *p, int slot)
{
    if (p->slot_key.empty() || p->slot_key[slot] == kNoKey) return;
    p->host_tier[p->slot_key[slot]].slot = -1;
    p->slot_key[slot] = kNoKey;
    p->slot_tick[slot] = 0;
}

bool slot_is_held(const lora_pool *p, int slot)
{
    return !p->slot_key.empty() && p->slot_pins[slot] > 0;
}

void destroy_host_tier(lora_pool *p)
{
    for (auto &kv : p->host_tier) {
        if (kv.second.A) cudaFreeHost(kv.second.A);
        if (kv.second.B) cudaFreeHost(kv.second.B);
    }
    p->host_tier.clear();
}

}  // namespace lora

extern "C" {

lora_status lora_host_register(lora_pool_t p, int64_t key, const void *A, const void *B, int rank,
                               float alpha)
{
    if (!p || !A || !B || key == kNoKey) return LORA_ERR_ARG;
    if (rank < 1 || rank > p->max_rank) return LORA_ERR_RANK;
    if (p->host_tier.count(key)) return LORA_ERR_SLOT_OCCUPIED;
    lora_status st = ensure_tier(p);
    if (st != LORA_OK) return st;
    HostAdapter h;
    const size_t a_bytes = (size_t)p->d_in * rank * 2, b_bytes = (size_t)rank * p->d_out * 2;
    if (cudaHostAlloc(&h.A, a_bytes, cudaHostAllocDefault) != cudaSuccess ||
        cudaHostAlloc(&h.B, b_bytes, cudaHostAllocDefault) != cudaSuccess) {
        cudaGetLastError();
        if (h.A) cudaFreeHost(h.A);
        if (h.B) cudaFreeHost(h.B);
        return LORA_ERR_OOM;
    }
    // A and B may be host or device memory
    if (cudaMemcpy(h.A, A, a_bytes, cudaMemcpyDefault) != cudaSuccess ||
        cudaMemcpy(h.B, B, b_bytes, cudaMemcpyDefault) != cudaSuccess) {
        cudaGetLastError();
        cudaFreeHost(h.A);
        cudaFreeHost(h.B);
        return LORA_ERR_CUDA;
    }
    h.rank = rank;
    h.alpha = alpha;
    p->host_tier[key] = h;
    return LORA_OK;
}

lora_status lora_host_unregister(lora_pool_t p, int64_t key)
{
    if (!p) return LORA_ERR_ARG;
    auto it = p->host_tier.find(key);
    if (it == p->host_tier.end()) return LORA_ERR_ARG;
    HostAdapter &h = it->second;
    if (h.slot >= 0) {
        if (p->slot_pins[h.slot] > 0 || p->chain_refs[h.slot] > 0) return LORA_ERR_IN_USE;
        lora_status st = evict(p, h.slot);
        if (st != LORA_OK) return st;
    }
    // an enqueued swap-in may still read the pinned copies
    CUDA_TRY(cudaEventSynchronize(p->ev_copy));
    cudaFreeHost(h.A);
    cudaFreeHost(h.B);
    p->host_tier.erase(it);
    return LORA_OK;
}

lora_status lora_acquire(lora_pool_t p, int64_t key, lora_stream_t stream, int *slot_out)
{
    if (!p || !slot_out) return LORA_ERR_ARG;
    auto it = p->host_tier.find(key);
    if (it == p->host_tier.end()) return LORA_ERR_ARG;
    HostAdapter &h = it->second;
    if (h.slot < 0) {
        lora_status st = swap_in(p, key, h);
        if (st != LORA_OK) return st;
        p->cache_misses += 1;
    } else {
        p->cache_hits += 1;
    }
    p->slot_pins[h.slot] += 1;
    p->slot_tick[h.slot] = ++p->tick;
    // the caller's next layer call must see the copy (this one, or a prefetch's)
    CUDA_TRY(cudaStreamWaitEvent((cudaStream_t)stream, p->ev_copy, 0));
    *slot_out = h.slot;
    return LORA_OK;
}

lora_status lora_prefetch(lora_pool_t p, int64_t key)
{
    if (!p) return LORA_ERR_ARG;
    auto it = p->host_tier.find(key);
    if (it == p->host_tier.end()) return LORA_ERR_ARG;
    HostAdapter &h = it->second;
    if (h.slot < 0) {
        lora_status st = swap_in(p, key, h);
        if (st != LORA_OK) return st;
    }
    p->slot_tick[h.slot] = ++p->tick;
    return LORA_OK;
}

lora_status lora_release(lora_pool_t p, int slot)
{
    if (!p) return LORA_ERR_ARG;
    if (slot < 0 || slot >= p->max_adapters) return LORA_ERR_SLOT_RANGE;
    if (p->slot_key.empty() || p->slot_key[slot] == kNoKey || p->slot_pins[slot] == 0)
        return LORA_ERR_ARG;
    p->slot_pins[slot] -= 1;
    return LORA_OK;
}

lora_status lora_cache_stats(lora_pool_t p, int64_t *out)
{
    if (!p || !out) return LORA_ERR_ARG;
    int64_t resident = 0;
    for (int64_t k : p->slot_key)
        if (k != kNoKey) ++resident;
    out[0] = (int64_t)p->host_tier.size();
    out[1] = resident;
    out[2] = p->cache_hits;
    out[3] = p->cache_misses;
    out[4] = p->cache_evictions;
    return LORA_OK;
}

}  // extern "C"
