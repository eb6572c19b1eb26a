// device_common.cuh -- sm_103a building blocks written as inline PTX:
// mbarriers with bounded waits, TMA tile loads, tcgen05 (TMEM allocation,
// MMA, commit, loads) and the shared-memory matrix descriptors they take.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "internal.h"

namespace lora {

// ------------------------------------------------------------------ generic

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Measurement hook of one launch (kTraceWords words, no-op for nullptr), global timer
// in ns: [0] the earliest CTA entry (atomic min), [1] the latest CTA exit (atomic
// max), [2] / [3] the earliest / latest moment a CTA got past its wait on the
// previous kernel in the stream (programmatic dependent launch; a kernel launched
// without it stamps its entry there). A CTA stamps its exit once all its threads are
// past their work; the caller of trace_release is the CTA's one thread that waits.
constexpr int kTraceWords = 4;

__device__ __forceinline__ void trace_stamp_min(uint64_t *w)
{
    atomicMin(reinterpret_cast<unsigned long long *>(w), (unsigned long long)global_timer_ns());
}

__device__ __forceinline__ void trace_stamp_max(uint64_t *w)
{
    atomicMax(reinterpret_cast<unsigned long long *>(w), (unsigned long long)global_timer_ns());
}

__device__ __forceinline__ void trace_enter(uint64_t *trace)
{
    if (trace && threadIdx.x == 0) trace_stamp_min(trace);
}

__device__ __forceinline__ void trace_release(uint64_t *trace)
{
    if (trace) {
        trace_stamp_min(trace + 2);
        trace_stamp_max(trace + 3);
    }
}

// Entry and release together: kernels that do not wait on the previous kernel.
__device__ __forceinline__ void trace_enter_released(uint64_t *trace)
{
    if (trace && threadIdx.x == 0) {
        trace_stamp_min(trace);
        trace_release(trace);
    }
}

__device__ __forceinline__ void trace_exit(uint64_t *trace)
{
    if (trace && threadIdx.x == 0) trace_stamp_max(trace + 1);
}

// Two packed bf16 -> fp32 (exact widening).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// sum_i a[i] * b[i] over 8 bf16 pairs packed in two uint4, accumulated into acc.
__device__ __forceinline__ float dot8_bf16(const uint4 &a, const uint4 &b, float acc)
{
    acc = fmaf(bf16_lo(a.x), bf16_lo(b.x), acc);
    acc = fmaf(bf16_hi(a.x), bf16_hi(b.x), acc);
    acc = fmaf(bf16_lo(a.y), bf16_lo(b.y), acc);
    acc = fmaf(bf16_hi(a.y), bf16_hi(b.y), acc);
    acc = fmaf(bf16_lo(a.z), bf16_lo(b.z), acc);
    acc = fmaf(bf16_hi(a.z), bf16_hi(b.z), acc);
    acc = fmaf(bf16_lo(a.w), bf16_lo(b.w), acc);
    acc = fmaf(bf16_hi(a.w), bf16_hi(b.w), acc);
    return acc;
}

// acc += sum_j v[j] * b[j] with b = 8 packed bf16.
__device__ __forceinline__ float dot8_f32_bf16(const float *v, const uint4 &b, float acc)
{
    acc = fmaf(v[0], bf16_lo(b.x), acc);
    acc = fmaf(v[1], bf16_hi(b.x), acc);
    acc = fmaf(v[2], bf16_lo(b.y), acc);
    acc = fmaf(v[3], bf16_hi(b.y), acc);
    acc = fmaf(v[4], bf16_lo(b.z), acc);
    acc = fmaf(v[5], bf16_hi(b.z), acc);
    acc = fmaf(v[6], bf16_lo(b.w), acc);
    acc = fmaf(v[7], bf16_hi(b.w), acc);
    return acc;
}

// Eight 4-bit codes (w: code j in bits 4j..4j+3, the lowest first) to the eight bf16
// values bf16(s * (q_j - z)), as four bf16x2 words in element order. 128 + q is exact
// in bf16 (bits 0x4300 | q), so (128 + q) - (128 + z) is the exact integer q - z, and
// one bf16 multiply rounds the exact product s (q - z) to nearest, ties to even.
// zz holds 128 + z twice, ss the scale twice.
__device__ __forceinline__ uint4 dequant8_q4(uint32_t w, __nv_bfloat162 zz, __nv_bfloat162 ss)
{
    // byte j of w: input 2j in the low nibble, 2j + 1 in the high one
    const uint32_t x = w & 0x0F0F0F0Fu, y = (w >> 4) & 0x0F0F0F0Fu;
    const uint32_t t01 = __byte_perm(x, y, 0x5140);  // q0 q1 q2 q3 as bytes
    const uint32_t t23 = __byte_perm(x, y, 0x7362);  // q4 q5 q6 q7
    const uint32_t bits[4] = {__byte_perm(t01, 0x43u, 0x4140), __byte_perm(t01, 0x43u, 0x4342),
                              __byte_perm(t23, 0x43u, 0x4140), __byte_perm(t23, 0x43u, 0x4342)};
    uint32_t o[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {  // bf16 pairs (128 + q_2p, 128 + q_2p+1)
        __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162 *>(&bits[p]);
        v = __hmul2(__hsub2(v, zz), ss);
        o[p] = *reinterpret_cast<const uint32_t *>(&v);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// 128 + z (z a 4-bit zero point) twice, and a bf16 scale twice, as bf16x2.
__device__ __forceinline__ __nv_bfloat162 q4_zero_pair(uint32_t z)
{
    const uint32_t bits = (0x4300u | z) * 0x10001u;
    return *reinterpret_cast<const __nv_bfloat162 *>(&bits);
}

__device__ __forceinline__ __nv_bfloat162 q4_scale_pair(uint16_t s)
{
    const uint32_t bits = (uint32_t)s * 0x10001u;
    return *reinterpret_cast<const __nv_bfloat162 *>(&bits);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);  // round to nearest even
    return *reinterpret_cast<uint32_t *>(&h);
}

// Fetch the line holding p into L2 (no register result).
__device__ __forceinline__ void prefetch_l2(const void *p)
{
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Bulk prefetch of `bytes` bytes at p into L2 (both multiples of 16): one request,
// carried out by the copy engine, not by the issuing thread's load slots.
__device__ __forceinline__ void prefetch_l2_bulk(const void *p, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void *p)
{
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// ------------------------------------------------- checked build (LORA_CHECK)
//
// Built with LORA_CHECK defined, every index a kernel gathers through a table is
// tested before use: out of range, it sets kErrRangeBit in the error word and is
// replaced by a safe one (the zero page, token 0, ...); otherwise these compile to
// nothing. The result of a call that met such an index is unspecified, but no access
// leaves its buffer.
#ifdef LORA_CHECK
__device__ __forceinline__ bool check_range(int v, int lo, int hi, int *err)
{
    if (v >= lo && v < hi) return true;
    if (err) atomicOr(err, kErrRangeBit);
    return false;
}
#define LORA_CHECKED(v, lo, hi, err, safe) (check_range((v), (lo), (hi), (err)) ? (v) : (safe))
#else
#define LORA_CHECKED(v, lo, hi, err, safe) (v)
#endif

// Is `id` a loaded slot of the table?  (rank field > 0)
__device__ __forceinline__ bool slot_loaded(const int32_t *slots, int slot_stride,
                                            int max_adapters, int id)
{
    return id >= 0 && id < max_adapters && slots[(size_t)id * slot_stride + SLOT_RANK] > 0;
}

// ----------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Wait for the phase with `parity` to complete, for at most limit_ns.
// Returns false (after raising the CTA's abort flag and, when err is not null,
// the pool's timeout bit) if it runs out, or if another role of the CTA has
// already aborted. Inlined: for loops that wait once per pipeline unit.
__device__ __forceinline__ bool mbar_wait_inl(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                             int *err, uint64_t limit_ns = kWaitTimeoutNs)
{
    if (mbar_try_wait(bar, parity)) return true;
    uint64_t start = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255u) == 0) {
            if (*abort_flag) return false;
            if (global_timer_ns() - start > limit_ns) {
                *abort_flag = 1;
                if (err) atomicOr(err, kErrTimeoutBit);
                return false;
            }
        }
    }
}

// The same wait out of line (most call sites: keeps the kernels' code small).
static __device__ __noinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                       int *err, uint64_t limit_ns = kWaitTimeoutNs)
{
    return mbar_wait_inl(bar, parity, abort_flag, err, limit_ns);
}

// ---------------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// 2-D tiled load of the box at (x = inner coordinate, y = row) into smem;
// completion is counted in bytes on `bar`. Out-of-range elements read zero.
__device__ __forceinline__ void tma_load_2d(void *smem_dst, const CUtensorMap *map, uint64_t *bar,
                                            int x, int y)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(map), "r"(smem_u32(bar)), "r"(x), "r"(y)
        : "memory");
}

// Same, with an L2 eviction-priority hint (cache policy from createpolicy).
__device__ __forceinline__ void tma_load_2d_hint(void *smem_dst, const CUtensorMap *map,
                                                 uint64_t *bar, int x, int y, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(smem_dst)),
        "l"(map), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 1-D bulk copy global -> shared (both 16-byte aligned, bytes a multiple of 16),
// completion counted in bytes on `bar`.
__device__ __forceinline__ void bulk_load(void *smem_dst, const void *gsrc, uint32_t bytes,
                                          uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(smem_dst)),
        "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// 2-D tiled store of the box at (x = inner coordinate, y = row) from shared memory
// (parts of the box outside the tensor are not written), as one bulk async-group.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, const void *smem_src, int x, int y)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(map),
                 "r"(smem_u32(smem_src)), "r"(x), "r"(y)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until this thread's bulk stores have finished reading their shared memory.
__device__ __forceinline__ void bulk_wait_read_all()
{
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Wait until this thread's bulk stores have completed.
__device__ __forceinline__ void bulk_wait_all()
{
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Make generic-proxy shared-memory writes visible to the async proxy
// (tensor cores / TMA) before signalling them.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ tcgen05

__device__ __forceinline__ void tmem_alloc(uint32_t *smem_result, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(smem_result)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulate; issued by one thread.
__device__ __forceinline__ void mma_bf16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every MMA this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint64_t *bar)
{
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// Instruction descriptor, kind::f16: bf16 A and B (both K-major), fp32 D, M x N.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N)
{
    return (1u << 4)                              // D format: f32
           | (1u << 7)                            // A format: bf16
           | (1u << 10)                           // B format: bf16
           | ((uint32_t)(N >> 3) << 17)           // N / 8
           | ((uint32_t)(M >> 4) << 24);          // M / 16
}

// Shared-memory matrix descriptor for a K-major operand stored in the
// 128-byte swizzle layout (rows of 64 bf16 = 128 B, groups of 8 rows 1024 B
// apart), as a TMA load with CU_TENSOR_MAP_SWIZZLE_128B writes it. The tile
// base must be 1024-byte aligned; stepping K inside the row adds bytes to
// the start address.
__device__ __forceinline__ uint64_t sdesc_k_sw128(uint32_t smem_addr)
{
    uint64_t d = 0;
    d |= (uint64_t)((smem_addr & 0x3FFFFu) >> 4);  // start address
    d |= (uint64_t)1 << 16;                         // leading byte offset (unused here)
    d |= (uint64_t)(1024 >> 4) << 32;               // stride byte offset: 8-row group pitch
    d |= (uint64_t)1 << 46;                         // descriptor version (sm_100 family)
    d |= (uint64_t)2 << 61;                         // swizzle: 128 B
    return d;
}

// Shared-memory matrix descriptor for a K-major operand without swizzle: core
// matrices of 8 rows x 16 bytes (128 contiguous bytes), `lbo` bytes between the
// core matrices that follow each other along K, `sbo` bytes between 8-row groups
// along M/N. The interleaved B pages ([n][8 rank rows] per page) are exactly
// this layout with sbo = 128 and lbo = the distance between two page slices.
__device__ __forceinline__ uint64_t sdesc_k_none(uint32_t smem_addr, uint32_t lbo, uint32_t sbo)
{
    uint64_t d = 0;
    d |= (uint64_t)((smem_addr & 0x3FFFFu) >> 4);  // start address
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;   // leading (K) byte offset
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;   // stride (M/N) byte offset
    d |= (uint64_t)1 << 46;                         // descriptor version (sm_100 family)
    return d;                                       // swizzle: none
}

// 32 TMEM lanes x 32 bit, N consecutive columns -> N registers per thread,
// followed by tcgen05.wait::ld inside the same asm block so the registers are
// never read before the load has landed.
__device__ __forceinline__ void tmem_ld16_wait(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_ld32_wait(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// ------------------------------------------- CTA pairs (cluster of two, cta_group::2)

__device__ __forceinline__ uint32_t cluster_cta_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// All threads of every CTA of the cluster (release / acquire at cluster scope).
__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The shared::cluster address of the same shared variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_map(const void *p, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}

// Arrive on an mbarrier given by its shared::cluster address (release at cluster scope).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t *bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// mbar_wait for a barrier that the other CTA of the pair signals (acquire at cluster
// scope); the same bound and abort behaviour.
static __device__ __noinline__ bool mbar_wait_cluster(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                               int *err, uint64_t limit_ns = kWaitTimeoutNs)
{
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t start = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if ((i & 255u) == 0) {
            if (*abort_flag) return false;
            if (global_timer_ns() - start > limit_ns) {
                *abort_flag = 1;
                if (err) atomicOr(err, kErrTimeoutBit);
                return false;
            }
        }
    }
}

// 2-D tiled load into this CTA's shared memory whose completion is counted on an
// mbarrier of either CTA of the pair (given by its shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void *smem_dst, const CUtensorMap *map, uint32_t bar_cluster,
                                                 int x, int y)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(map), "r"(bar_cluster), "r"(x), "r"(y)
        : "memory");
}

// TMEM allocation shared by the pair: one warp of each CTA executes these.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t *smem_result, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(smem_result)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// D[tmem of both CTAs] (+)= A * B^T over the pair: M = 256 rows, rows 0-127 from CTA 0's
// A tile and TMEM, 128-255 from CTA 1's; B's N columns split in halves the same way.
// Issued by one thread of CTA 0 with descriptors of its own shared memory (the peer's
// tiles sit at the same offsets).
__device__ __forceinline__ void mma_bf16_ss_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                 uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` (same offset) in every CTA of `cta_mask` when the pair MMAs this
// thread issued so far have completed.
__device__ __forceinline__ void mma_commit_pair(uint64_t *bar, uint16_t cta_mask)
{
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(cta_mask)
        : "memory");
}

// ----------------------------------------------------------- named barriers

// Barrier `id` (1..15) over `count` threads (a multiple of 32); the calling
// warps wait.
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t count)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Arrive on barrier `id` without waiting for the others.
__device__ __forceinline__ void named_bar_arrive(uint32_t id, uint32_t count)
{
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}


// ------------------------------------------------ programmatic dependent launch

// Let the next kernel in the stream start its prologue now.
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Wait until the previous kernel in the stream has completed and its memory
// is visible (no-op when launched without the programmatic attribute).
__device__ __forceinline__ void pdl_wait_prior()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace lora
