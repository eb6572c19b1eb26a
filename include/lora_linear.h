/*
 * lora_linear.h -- C ABI of the GB300 (sm_103a) heterogeneous multi-LoRA linear layer.
 *
 * The layer: for a batch of T tokens, each tagged with an adapter slot id
 * (-1 = base only),
 *
 *     Y[t,:] = X[t,:] W_base^T + (alpha_i / r_i) (X[t,:] A_i) B_i,   i = ids[t]
 *
 * with A_i d_in x r_i and B_i r_i x d_out, over adapters resident in one GPU
 * pool. Definition: "LoRA-Land: 将大模型变成操作系统..." (blog), section
 * 核心实现解析 / 2. 多 LoRA 批处理调度 (shared base weight, per-group A,B
 * correction, X@A formed first as a low-dimensional intermediate; the printed
 * equation's transposes are garbled, the row-token reading above is used);
 * "多 LoRA 热插拔: 一模型服多租户" (vLLM tutorial), sections "LoRA 速览"
 * (W'x = Wx + BAx) and "vLLM 的 Multi-LoRA 怎么实现" (one unified adapter
 * memory pool; different adapters in one batch; the base path always shared);
 * icman.com.cn Multi-LoRA article, section 3.2 (alpha controls the scale,
 * read as s = alpha / rank).
 *
 * Conventions for every call:
 *  - bf16 tensors are passed as raw pointers to bfloat16 values, row-major,
 *    densely packed. X is T x d_in, W_base is d_out x d_in (the nn.Linear
 *    layout), Y is T x d_out. d_in and d_out must be multiples of 8 and
 *    X, W_base, Y 16-byte aligned (any cudaMalloc / torch allocation is).
 *  - Device pointers are CUDA device (or managed) memory of the pool's device.
 *  - Every call returns a lora_status; a call that returns an error has
 *    enqueued no GPU work and changed no pool state.
 *  - A pool is not thread-safe: use it from one host thread at a time.
 *  - Only GB300-class devices (compute capability 10.3) are supported; on any
 *    other device lora_pool_create returns LORA_ERR_UNSUPPORTED. There is no
 *    CPU fall-back.
 *  - The library is also built with LORA_CHECK defined (liblora_linear_check.so,
 *    the same ABI): there every index a kernel gathers through a table (page
 *    ids, token positions, slot ids, segment and tile entries, split-K partial
 *    slots) is range-checked first; an index out of range sets the pool's error
 *    word (LORA_ERR_RANGE) and the access is skipped or redirected to the zero
 *    page, never made. It stands in for a memory checker and runs slower.
 */
#ifndef LORA_LINEAR_H
#define LORA_LINEAR_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LORA_ABI_VERSION 1

/* Opaque pool handle: owns the adapter page arenas, the slot table and all
 * scratch memory of the calls below. */
typedef struct lora_pool lora_pool;
typedef lora_pool *lora_pool_t;

/* A cudaStream_t (the same type, declared without the CUDA headers).
 * NULL means the legacy default stream. */
typedef struct CUstream_st *lora_stream_t;

typedef enum {
    LORA_OK = 0,
    LORA_ERR_ARG = 1,             /* null pointer, negative size, bad option   */
    LORA_ERR_SHAPE = 2,           /* d_in / d_out not a positive multiple of 8,
                                     or beyond the limits below               */
    LORA_ERR_SLOT_RANGE = 3,      /* slot outside [0, max_adapters)            */
    LORA_ERR_SLOT_OCCUPIED = 4,   /* load into a slot that holds an adapter    */
    LORA_ERR_SLOT_EMPTY = 5,      /* unload of an empty slot                   */
    LORA_ERR_RANK = 6,            /* rank outside [1, max_rank]                */
    LORA_ERR_BAD_ADAPTER_ID = 7,  /* a token id was neither -1 nor a loaded slot
                                     (reported by lora_pool_check_errors)      */
    LORA_ERR_CUDA = 8,            /* a CUDA runtime call failed                */
    LORA_ERR_OOM = 9,             /* device allocation failed                  */
    LORA_ERR_TIMEOUT = 10,        /* a kernel's bounded wait ran out (reported
                                     by lora_pool_check_errors)                */
    LORA_ERR_UNSUPPORTED = 11,    /* no compute-capability-10.3 device         */
    LORA_ERR_IN_USE = 12,         /* unload of an adapter a chain still lists  */
    LORA_ERR_RANGE = 13           /* a kernel of the checked build (LORA_CHECK)
                                     met an index outside its table or buffer
                                     (reported by lora_pool_check_errors)      */
} lora_status;

/* Limits. */
#define LORA_MAX_ADAPTERS 4096    /* slots per pool                            */
#define LORA_MAX_RANK 256         /* largest rank a pool can hold              */
#define LORA_MAX_DIM 65536        /* largest d_in / d_out                      */
#define LORA_RANK_PAGE 8          /* rank rows per pool page                   */
#define LORA_MAX_GROUP 8          /* layers of one lora_linear_grouped call    */

/* Which kernel family lora_linear uses. AUTO picks DECODE for T <= 256, the DECODE
 * kernels over consecutive slices of 256 tokens for 256 < T <= 512, and PREFILL
 * above; a forced DECODE accepts T <= 256 only. All compute the same result (up to
 * the order of the fp32 sums). */
typedef enum { LORA_PATH_AUTO = 0, LORA_PATH_DECODE = 1, LORA_PATH_PREFILL = 2 } lora_path;

/* Which prefill GEMM kernel the PREFILL path uses. AUTO picks PAIR for T > 128:
 * a cluster of two CTAs per 256-token x 256-column tile (tcgen05 MMAs spanning
 * both SMs); SINGLE is one CTA per 128 x 256 tile. Both compute the same result. */
typedef enum { LORA_PREFILL_AUTO = 0, LORA_PREFILL_SINGLE = 1, LORA_PREFILL_PAIR = 2 } lora_prefill_kernel;

/*
 * Create a pool on the current CUDA device for one linear layer of shape
 * d_in -> d_out, with room for max_adapters adapters of rank <= max_rank.
 *
 * The unified adapter pool of the vLLM tutorial ("vLLM 的 Multi-LoRA 怎么实现",
 * item 1) and the LoRA-Land blog (技术方案: only the A,B matrices are added per
 * adapter). Memory is paged at rank granularity: each page holds 8 rank rows
 * of one adapter (8 columns of A, stored transposed as 8 x d_in, and 8 rows
 * of B, stored interleaved as d_out x 8); an adapter of rank r holds ceil(r/8)
 * pages taken from a free list. All page arenas, the slot table and the error
 * word are allocated here, once: loading and unloading never allocate. The
 * arenas hold max_adapters * ceil(max_rank/8) pages, a zero page and a reserve
 * of 2 * ceil(max_rank/8) pages (see lora_load_adapter).
 * Scratch for lora_linear is sized by lora_pool_reserve (or grown by the
 * first call with a larger T).
 *
 * Returns LORA_ERR_SHAPE for bad dimensions, LORA_ERR_RANK for max_rank
 * outside [1, LORA_MAX_RANK], LORA_ERR_ARG for max_adapters outside
 * [1, LORA_MAX_ADAPTERS] or out == NULL, LORA_ERR_OOM if the arenas do not
 * fit, LORA_ERR_UNSUPPORTED on a device that is not compute capability 10.3.
 * On success *out owns everything; release it with lora_pool_destroy.
 */
lora_status lora_pool_create(int max_adapters, int max_rank, int d_in, int d_out,
                             lora_pool_t *out);

/* Wait for the device to finish all work (every stream: graph replays that
 * use the pool are not tracked), then free all of the pool's device memory.
 * The handle is invalid afterwards. NULL returns LORA_ERR_ARG. The pages have
 * no counterpart for this call beyond the unified pool itself (vLLM tutorial,
 * "vLLM 的 Multi-LoRA 怎么实现", item 1): it is the pool's destructor. */
lora_status lora_pool_destroy(lora_pool_t pool);

/*
 * Size the per-call scratch for batches of up to max_tokens tokens (segment
 * tables, the fp32 low-rank intermediate, split-K partial sums, host-call
 * staging). Calls with larger T grow it on first use, which allocates and
 * synchronises the device: call this first when lora_linear will run inside a
 * CUDA graph capture.
 */
lora_status lora_pool_reserve(lora_pool_t pool, int max_tokens);

/*
 * Load an adapter into an empty slot ("load_adapter" of the LoRA-Land blog,
 * 热插拔 API: A,B are moved to the GPU and indexed; the vLLM tutorial's
 * 动态上下线: adapters come and go without restarting).
 *   A: bf16, d_in x rank, row-major.  B: bf16, rank x d_out, row-major.
 *   Host or device pointers (detected); the data is copied into pool pages
 *   and the caller keeps ownership (it may free A,B on return). Device data
 *   must be complete before the call (no stream ordering is applied).
 *   alpha: the adapter's scale numerator; the pool stores s = alpha / rank
 *   (fp32), rank being the rank passed here.
 * Ordering without a device-wide stall (icman.com.cn Multi-LoRA article,
 * section 4.2: a cold adapter load must not hold up the requests already
 * running): the call waits on the host only for its own copy of A and B into
 * pool-owned memory and, when the pool has pages that no enqueued layer call
 * can still read, for writing those pages. (Pages an unload frees become such
 * once the calls enqueued before it have run; the reserve of lora_pool_create
 * lets a swap on a full pool find them.) Otherwise the pages are written on
 * the pool's internal copy stream after every layer call already enqueued on
 * this pool. The table row always is (on any stream, those calls keep seeing
 * the old state), and every layer call enqueued on the pool after the return
 * waits for it on the GPU. Other
 * streams and other pools are not held up (on the GPU, the changes of a pool
 * used on the legacy default stream also follow other streams' earlier work:
 * see lora_pool_check_errors). Calls replayed from a CUDA graph
 * are not tracked: a graph that uses the pool must have finished (or be
 * ordered by the caller) before a load, unload or chain definition, and
 * changes must be made before the capture.
 * Loading into an occupied slot is an error: a hot swap is unload, then load.
 * Errors: SLOT_RANGE, SLOT_OCCUPIED, RANK, ARG (null A/B), OOM (no free
 * pages), CUDA.
 */
lora_status lora_load_adapter(lora_pool_t pool, int slot, const void *A, const void *B,
                              int rank, float alpha);

/* Unload ("unload_adapter", same sections): returns the slot's pages to the
 * free list and marks it empty. Ordered like a load, without waiting on the
 * host: calls enqueued on the pool before it still see the adapter, calls
 * enqueued after it see an empty slot (an id naming it is then a bad id).
 * Unloading a chain slot releases its members and frees no pages; unloading a
 * slot the host tier filled drops it from the cache (the key stays registered).
 * Errors: SLOT_RANGE, SLOT_EMPTY, IN_USE (a chain still lists the adapter, or
 * it is acquired from the host tier). */
lora_status lora_unload_adapter(lora_pool_t pool, int slot);

/*
 * Adapter chain: make chain_slot stand for the n adapters in member_slots
 * applied together, so that a token with id chain_slot gets
 *
 *     Y[t] = X[t] W_base^T + sum over members m of s_m (X[t] A_m) B_m.
 *
 * The LoRA-Land blog combines adapters like a pipeline applied to the kernel
 * in order (section 技术方案 item 3; section 核心实现解析 / 3. 热插拔 API 与组合,
 * set_adaptive_chain); at one linear layer the members' weight updates add,
 * W + dW_1 + ... + dW_n, whatever their order. The chain copies no weights:
 * its slot lists the members' pages, each with its member's scale, so both
 * kernel families run it as one adapter of rank sum(r_m).
 *   member_slots: HOST array of n >= 1 distinct slots that hold adapters (not
 *   chains); their pages together must fit one slot (sum of ceil(r_m / 8)
 *   pages <= ceil(max_rank / 8)). chain_slot must be empty.
 * Ordered like a load (calls enqueued before it see an empty chain slot). While
 * a chain lists an adapter, unloading that adapter fails with IN_USE.
 * Errors: ARG (null list, n < 1, a repeated member, a member that is itself a
 * chain or the chain slot), SLOT_RANGE, SLOT_OCCUPIED (chain_slot), SLOT_EMPTY
 * (a member), RANK (the pages do not fit), CUDA.
 */
lora_status lora_define_chain(lora_pool_t pool, int chain_slot, const int *member_slots, int n);

/*
 * The hot path. For every token t: Y[t] = X[t] W_base^T + s_i (X[t] A_i) B_i
 * with i = token_adapter_ids[t]; id -1 gives the base product only (the vLLM
 * tutorial's 按请求切换 LoRA: no adapter -> pure base). Prefill-sized batches
 * are grouped by adapter with a stable sort ("Grouped Multi-LoRA Execution",
 * LoRA-Land blog section 2); decode-sized batches (T <= 256) gather each
 * token's adapter pages directly. The low-rank intermediate X A_i is kept in
 * fp32 (decode) or as an fp32-accurate bf16 hi + lo pair (prefill), and the
 * result is rounded to bf16 once.
 *   X: device bf16 T x d_in.  W_base: device bf16 d_out x d_in.
 *   token_adapter_ids: device int32[T].  Y: device bf16 T x d_out (written
 *   once; must not alias X or W_base).  T >= 0 (T == 0 does nothing).
 * Asynchronous: enqueued on `stream`, returns without waiting. X, W_base and
 * the ids must stay valid until the stream reaches the call.
 * Stream order: the decode kernels are launched with programmatic dependent
 * launch and may start while the kernel before them in the stream still runs.
 * X, the ids, Y and the pool's state are used in stream order; W_base, being a
 * weight, is already read before that wait. A kernel that writes W_base must
 * therefore not be the one directly before the call when it lets dependent
 * kernels launch early (griddepcontrol.launch_dependents) before writing it;
 * a copy, an event wait or any ordinary kernel in between keeps the order.
 * Ids that are neither -1 nor a loaded slot do not fall back silently (the
 * icman.com.cn article's section 4.1, strict mode): the kernels set the
 * pool's device error word, and the next lora_pool_check_errors returns
 * LORA_ERR_BAD_ADAPTER_ID. Such rows of Y are unspecified; other rows stay
 * correct.
 * Errors returned at once: ARG (null pointers, T < 0, T > 256 with a forced
 * DECODE path), OOM (scratch growth failed), CUDA.
 */
lora_status lora_linear(lora_pool_t pool, const void *X, const void *W_base,
                        const int32_t *token_adapter_ids, int T, void *Y,
                        lora_stream_t stream);

/*
 * Host tier. More adapters than the pool's slots can be registered under
 * 64-bit keys; the pool keeps pinned host copies and caches the active ones on
 * the GPU, swapping the least recently used one out when a missing adapter is
 * needed (icman.com.cn Multi-LoRA article, sections 2.1-2.2: adapters kept in
 * host memory, the active ones cached on the GPU, LRU swap-out; the vLLM
 * tutorial's "max-loras vs max-cpu-loras": a GPU set backed by a CPU set).
 * A swap-in is asynchronous: it is enqueued on the pool's copy stream after
 * every layer call already enqueued on the pool (on any stream) and never
 * blocks the host, and the acquiring stream waits for it (the same article's section 4.2: cold loads
 * must not stall the requests already running). The tier takes empty slots
 * (from the highest index down) and evicts only slots it filled itself with
 * no acquisition outstanding and no chain listing them; manually loaded slots
 * are never evicted. Calls captured into a CUDA graph are not ordered against
 * swap-ins: acquire before capturing, and keep the slots acquired while the
 * graph replays.
 */

/* Register an adapter in the host tier: A, B (host or device pointers, the
 * lora_load_adapter layouts) are copied into pool-owned pinned memory.
 * Host-blocking. Errors: ARG (null pointers, key INT64_MIN), RANK,
 * SLOT_OCCUPIED (the key is taken), OOM, CUDA. */
lora_status lora_host_register(lora_pool_t pool, int64_t key, const void *A, const void *B,
                               int rank, float alpha);

/* Remove a key from the host tier (evicting it from the GPU if resident).
 * Errors: ARG (unknown key), IN_USE (acquired, or listed by a chain), CUDA. */
lora_status lora_host_unregister(lora_pool_t pool, int64_t key);

/* Make `key` resident and hold it: *slot_out receives its slot id for
 * token_adapter_ids. On a miss the least recently used unheld cached adapter
 * may be evicted and the swap-in is enqueued; `stream` is made to wait for the
 * copy, so layer calls enqueued on it afterwards see the adapter. Each acquire
 * needs a lora_release. Errors: ARG (unknown key, null slot_out), OOM (every
 * slot or page is held), CUDA. */
lora_status lora_acquire(lora_pool_t pool, int64_t key, lora_stream_t stream, int *slot_out);

/* Start the swap-in of `key` without holding it (a hot adapter named ahead of
 * its requests); a later lora_acquire then hits. Errors: as lora_acquire. */
lora_status lora_prefetch(lora_pool_t pool, int64_t key);

/* Drop one hold on a slot returned by lora_acquire. The adapter stays cached
 * until it is evicted. Errors: SLOT_RANGE, ARG (not a held cached slot). */
lora_status lora_release(lora_pool_t pool, int slot);

/* out[5]: registered keys, resident cached adapters, hits, misses, evictions. */
#define LORA_CACHE_STATS_COUNT 5
lora_status lora_cache_stats(lora_pool_t pool, int64_t *out);

/*
 * Several LoRA linear layers that share one batch of token ids, in one launch
 * chain: for m = 0..n-1, Y[m] = lora_linear(pools[m], X[m], W_base[m], ids).
 * The layers are typically the target modules of one transformer layer (q, k,
 * v, o, gate, up, down), each module's adapters held in its own pool under the
 * same slot ids. The pages train one adapter over these seven projections
 * ("多 LoRA 热插拔: 一模型服多租户" (vLLM tutorial), sections "训练出 vLLM
 * 兼容的 LoRA" (target_modules) and "性能注意事项" (one target set for the
 * whole batch); icman.com.cn Multi-LoRA article, section 3.2); running them
 * in one launch chain answers the per-call dispatch cost that the same
 * article's section 4.2 names.
 *   n: 1..LORA_MAX_GROUP.  pools, X, W_base, Y: HOST arrays of n entries
 *   (pool handles and device pointers with the lora_linear layouts of each
 *   pool's d_in / d_out); the pools must be distinct and on one device.
 *   token_adapter_ids: device int32[T], shared by all layers.
 * Decode-sized batches (T <= 256, or pools[0] forced to DECODE) run all layers
 * in the same two kernels: one stream-K split over all the layers' weights, so
 * the device streams them as one workload. Larger batches run the layers one
 * after another, each as lora_linear would (pools[0]'s path setting applies).
 * Results equal those of n separate lora_linear calls up to the order of the
 * fp32 split-K sums. Bad ids are reported per pool (lora_pool_check_errors of
 * the layer's pool); a kernel timeout in pools[0]'s error word. Scratch: each
 * pool's per-token scratch, and pools[0] holds the call's split-K partial
 * sums (grown on first use of a larger group, after a device synchronise).
 * Errors returned at once: ARG (n out of range, null pointers, repeated or
 * cross-device pools, T < 0, T > 256 with a forced DECODE path), SHAPE, OOM,
 * CUDA.
 */
lora_status lora_linear_grouped(int n, const lora_pool_t *pools, const void *const *X,
                                const void *const *W_base, const int32_t *token_adapter_ids,
                                int T, void *const *Y, lora_stream_t stream);

/*
 * Same as lora_linear, but X, token_adapter_ids and Y are HOST pointers
 * (pinned memory gives full copy speed). The call copies X and the ids into
 * pool-owned device staging on `stream`, runs the layer, copies Y back and
 * waits for the stream before returning. W_base stays a device pointer (the
 * resident base weight).
 */
lora_status lora_linear_host(lora_pool_t pool, const void *X_host, const void *W_base,
                             const int32_t *ids_host, int T, void *Y_host,
                             lora_stream_t stream);

/*
 * Base product only, Y = X W_base^T, with the same GEMM kernels lora_linear
 * uses (the reference point the adapter overhead is measured against).
 * Same pointer and stream rules as lora_linear.
 */
lora_status lora_base_linear(lora_pool_t pool, const void *X, const void *W_base, int T,
                             void *Y, lora_stream_t stream);

/*
 * The layer over a 4-bit quantised base ("多 LoRA 热插拔: 一模型服多租户" (vLLM
 * tutorial), section 性能注意事项: a base quantised to 4 bits, AWQ-INT4, serves the
 * bf16 adapters unchanged). The pages give no format; this one is used:
 *   Wq: device bytes [d_out][d_in / 2], two unsigned 4-bit codes per byte along the
 *       input dimension (the even input in the low nibble): the nn.Linear layout;
 *   scales: device bf16 [d_in / 128][d_out], one per (group of 128 inputs, output row);
 *   zeros: device bytes [d_in / 128][d_out], the 4-bit zero points (0..15);
 *   W[n][k] = bf16(scales[k/128][n] * (q[n][k] - zeros[k/128][n])): the exact product,
 *   rounded once to bf16 (to nearest, ties to even), as a kernel that dequantises to
 *   the activation type before its bf16 product would. Then Y as lora_linear computes
 *   it, with the same ids, pool and rules. d_in must be a multiple of 128 and d_out of
 *   16 (the pool's shapes).
 * Decode-sized batches (T <= 256) stream the codes (a quarter of a bf16 base's bytes)
 * and dequantise W tiles in shared memory on the way to the tensor cores; larger batches
 * dequantise W into pool scratch (d_out x d_in bf16, allocated on the first such call,
 * which then synchronises like a scratch growth) and run the bf16 prefill path.
 * Wq, scales and zeros must start on 16-byte boundaries.
 * Errors: as lora_linear; SHAPE when d_in % 128 or d_out % 16 is not zero; ARG for a
 * pointer that is null or not 16-byte aligned.
 */
lora_status lora_linear_q4(lora_pool_t pool, const void *X, const void *Wq, const void *scales,
                           const void *zeros, const int32_t *token_adapter_ids, int T, void *Y,
                           lora_stream_t stream);

/* The base product over the 4-bit base only (no adapters; the reference point of the
 * adapters' overhead on that base). Same arguments and rules as lora_linear_q4. */
lora_status lora_base_linear_q4(lora_pool_t pool, const void *X, const void *Wq, const void *scales,
                                const void *zeros, int T, void *Y, lora_stream_t stream);

/* The 4-bit base (the format of lora_linear_q4, device pointers) dequantised to bf16
 * W [d_out][d_in], asynchronously on `stream`. Needs no pool.
 * Wq and W must start on 16-byte boundaries.
 * Errors: ARG (null or misaligned pointers), SHAPE (d_in not a multiple of 128, or a dimension
 * outside 8..LORA_MAX_DIM or not a multiple of 8), CUDA. */
lora_status lora_dequant_q4(const void *Wq, const void *scales, const void *zeros, int d_out, int d_in,
                            void *W, lora_stream_t stream);

/*
 * Base product Y = X W_base^T for callers that cannot allocate device memory.
 * The pages have no counterpart for this call: it exists for users of this
 * library who may not call cudaMalloc (code living inside another framework's
 * memory arena, plugins whose host forbids device allocation after start-up,
 * callers that must never block on an allocator). It needs no pool and
 * allocates nothing (no cudaMalloc, no cudaFree, no allocating library call):
 * the same decode kernels as lora_base_linear take their split-K scratch from
 * a fixed __device__ array compiled into the library (16 MiB: 4,194,304 fp32
 * partial sums), which every GPU that loads the library holds until the
 * process exits.
 *   X: device bf16 T x d_in, W_base: device bf16 d_out x d_in, Y: device bf16
 *   T x d_out; 0 <= T <= 256; d_in, d_out positive multiples of 8 up to
 *   LORA_MAX_DIM. Asynchronous on `stream`.
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, once per device, with that device current): make
 * that first call before any CUDA stream capture.
 * Every call shares the one array and leaves its contents behind; calls that
 * overlap on the GPU (other streams, or concurrent replays) race on it and
 * must be serialised by the caller.
 * Errors: ARG (null pointers, T outside [0, 256]), SHAPE (bad d_in / d_out,
 * or T x d_out too large for the fixed scratch). The partial sums take
 * G * S * T * 128 floats for G CTAs each touching at most S tiles of 128
 * output rows; when that exceeds the array the call runs with fewer CTAs,
 * down to one CTA over all ceil(d_out / 128) tiles, so it succeeds exactly
 * when ceil(d_out / 128) * 128 * T <= 4,194,304 (T = 256: d_out up to 16384;
 * T = 64: up to 65536). UNSUPPORTED (device not compute capability 10.3),
 * CUDA. A kernel wait that times out is not reported by this call (the
 * kernels are given no error word); its Y is then incomplete.
 */
lora_status lora_base_linear_noalloc(const void *X, const void *W_base, int T, int d_in,
                                     int d_out, void *Y, lora_stream_t stream);

/*
 * Strict-mode report (icman.com.cn Multi-LoRA article, section 4.1: an unknown
 * adapter must surface as an error, not fall back to the base output
 * silently). Waits for the layer calls enqueued on this pool (graph replays
 * are not tracked: synchronise their stream first), then reads and clears the
 * pool's device error word in one atomic step, so a bit set meanwhile by a
 * kernel on another stream is never lost. Other streams are not waited for,
 * with one exception that CUDA defines: an event recorded on the legacy
 * default stream (NULL) completes only after all earlier work of the context,
 * so the calls of a pool used on that stream also wait for other streams' work
 * enqueued before them.
 * Returns LORA_OK, LORA_ERR_BAD_ADAPTER_ID, LORA_ERR_TIMEOUT or LORA_ERR_RANGE
 * (the first of these present), or LORA_ERR_CUDA if the device reported an
 * error.
 */
lora_status lora_pool_check_errors(lora_pool_t pool);

/*
 * Test hook (host only, needs no GPU; no counterpart in the pages): the decode
 * path's plan for n layers of T tokens -- the stream-K split and the kernels'
 * resources -- as lora_linear / lora_linear_grouped would compute it with
 * num_sms SMs. d_in, d_out, max_pages: HOST arrays of n entries (max_pages 0:
 * no adapters). out[LORA_PLAN_INFO_COUNT] = {units, ranges G, CTAs launched,
 * most tiles per range, TMEM accumulators, pipeline stages, TMEM columns,
 * GEMM dynamic shared memory bytes, shrink pairs, finishing blocks, register-
 * bounded variant (0/1), T rounded up to 16, split-K partial floats, A pages
 * requested into L2 before the wait on the previous kernel (0/1)}.
 * Errors: ARG (null pointers, n outside 1..LORA_MAX_GROUP, T outside 1..256,
 * num_sms < 1), SHAPE.
 */
#define LORA_PLAN_INFO_COUNT 14
lora_status lora_decode_plan_info(int n, int T, const int *d_in, const int *d_out,
                                  const int *max_pages, int num_sms, int64_t *out);

/*
 * Test hook for the kernels' bounded waits (no counterpart in the pages): runs
 * one wait, with the same code the kernels use, on an mbarrier that nothing
 * completes. It gives up after limit_us microseconds (1..2,000,000), sets the
 * pool's timeout bit and returns; the next lora_pool_check_errors reports
 * LORA_ERR_TIMEOUT and the context stays usable. Every mbarrier wait in the
 * kernels is bounded this way (2 s): a lost arrival ends as an error status,
 * never as a hang. Asynchronous on `stream`. Errors: ARG, CUDA.
 */
lora_status lora_pool_selftest_wait(lora_pool_t pool, int limit_us, lora_stream_t stream);

/*
 * Test hook for stream order (no counterpart in the pages): one kernel that lets
 * the next kernel in the stream launch at once (programmatic dependent launch) and
 * only after delay_us microseconds (1..100,000) copies n int32 from src to dst (both
 * DEVICE pointers). A lora_linear enqueued right after it with dst as its ids must
 * still use the copied ids: its kernels may start early, but read stream-ordered
 * data only after their wait on the kernel before them. Asynchronous on `stream`.
 * Errors: ARG, CUDA.
 */
lora_status lora_test_delayed_copy(const int32_t *src, int32_t *dst, int n, int delay_us,
                                   lora_stream_t stream);

/*
 * Test hook: run only the segment builder of the prefill path -- the grouping
 * of a batch by adapter id of the LoRA-Land blog, section 核心实现解析 / 2.
 * 多 LoRA 批处理调度 ("Grouped Multi-LoRA Execution": the batch is grouped by
 * LoRA ID and each group run with its own A, B) -- on device ids[T] and copy its
 * tables out (device pointers): order[T] (token indices stably sorted by id,
 * base-only tokens first), *n_base, *num_seg, seg_start[num_seg + 1] (offsets
 * into order; seg_start[0] = n_base, seg_start[num_seg] = T) and
 * seg_slot[num_seg] (ascending slot ids). seg_start and seg_slot must have
 * room for min(T, max_adapters) + 1 entries. Ids that are neither -1 nor a
 * loaded slot are grouped with the base-only tokens and set the error word.
 */
lora_status lora_build_segments(lora_pool_t pool, const int32_t *ids, int T, int32_t *order,
                                int32_t *n_base, int32_t *num_seg, int32_t *seg_start,
                                int32_t *seg_slot, lora_stream_t stream);

/* Pool counters, written to out[0..LORA_STATS_COUNT):
 * loaded slots, free pages, total pages, loads, unloads, linear calls,
 * bytes of device memory held. Total pages = max_adapters * ceil(max_rank/8)
 * (the zero page and the reserve not counted); free pages = total pages minus
 * the pages loaded adapters hold. The counterpart in the pages is the startup
 * check of icman.com.cn Multi-LoRA article, section 4.1 (confirm from the logs
 * which adapters are loaded); the counters read the host mirror, no GPU work. */
#define LORA_STATS_COUNT 7
lora_status lora_pool_stats(lora_pool_t pool, int64_t *out);

/*
 * Measurement hook. While enabled, every lora_linear / lora_base_linear call
 * records CUDA events on its stream around each kernel it launches.
 * lora_pool_kernel_times waits for the last call and writes the device time
 * of each of its kernels in milliseconds to ms[0..LORA_KERNEL_SLOTS):
 *   0 segment builder, 1 shrink, 2 base GEMM (prefill: with the fused
 *   expand), 3 decode finishing pass (split-K sum + expand).
 * Slots a call did not use read 0.
 */
#define LORA_KERNEL_SLOTS 4
lora_status lora_pool_enable_timing(lora_pool_t pool, int enable);
lora_status lora_pool_kernel_times(lora_pool_t pool, float *ms);

/*
 * Measurement hook that keeps programmatic dependent launch intact (no events
 * between the kernels; no counterpart in the pages). While buf is set, the
 * k-th layer call on the pool after this call (k = 0, 1, ...; a grouped call
 * counts on its first pool) writes, for each kernel it launches, four global
 * timer values (ns) into
 *   buf[((k % n_calls) * LORA_KERNEL_SLOTS + slot) * 4 + {0, 1, 2, 3}]
 * (slots as for lora_pool_kernel_times): {0} its first CTA's entry (atomic
 * min), {1} its last CTA's exit (atomic max), {2, 3} the first and the last
 * moment a CTA got past its wait on the kernel before it in the stream (for a
 * kernel that does not wait, its CTAs' entries). The caller sets each group to
 * {UINT64_MAX, 0, UINT64_MAX, 0} before the calls and reads them after.
 * buf: DEVICE memory of n_calls * LORA_KERNEL_SLOTS * 4 uint64. Calls captured
 * into a CUDA graph keep the entries they were captured with. NULL turns it
 * off. Errors: ARG (n_calls < 1 with a buffer).
 */
lora_status lora_pool_set_trace(lora_pool_t pool, uint64_t *buf, int n_calls);

/* Force a kernel family (lora_path); LORA_PATH_AUTO restores the default. */
lora_status lora_pool_set_path(lora_pool_t pool, int path);

/* Force the prefill GEMM kernel (lora_prefill_kernel); LORA_PREFILL_AUTO restores
 * the default. Errors: ARG (unknown value), UNSUPPORTED (PAIR on a pool whose B arena
 * has 2^31 or more rows of 8 rank values). */
lora_status lora_pool_set_prefill_kernel(lora_pool_t pool, int kernel);

/* Static description of a status code. */
const char *lora_status_string(lora_status status);

/* LORA_ABI_VERSION of the built library. */
int lora_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LORA_LINEAR_H */
