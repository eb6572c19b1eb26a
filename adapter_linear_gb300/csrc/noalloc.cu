// noalloc.cu -- lora_base_linear_noalloc: the decode base product for callers
// that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at all: code running inside another
// framework's memory arena, plugins whose host forbids device allocation after
// start-up, or callers that must never synchronise on an allocator. This entry
// point runs the same two decode kernels as lora_base_linear (stream-K tcgen05
// GEMM + finishing pass) but takes their split-K scratch from a fixed array
// compiled into the library, so it allocates nothing: no cudaMalloc, no
// cudaFree, no allocating library call. It needs no pool either.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds it until the process exits. In host code its name is only a
// stand-in; the device address is looked up with cudaGetSymbolAddress once per
// device (with that device current) on the first call there, and cached.
#include <mutex>

#include "../../include/lora_linear.h"
#include "device_common.cuh"

namespace lora {
namespace {

// Split-K partial sums (G * max_seg * T * 128 floats per call): 16 MiB. The kernels
// get no error word here (a wait that times out is not reported by this entry point).
constexpr size_t kNoallocScratchFloats = (size_t)4 << 20;

static __device__ __align__(256) float g_noalloc_scratch[kNoallocScratchFloats];

constexpr int kMaxDevices = 64;

struct DeviceSetup {
    bool ready = false;
    float *scratch = nullptr;  // device address of g_noalloc_scratch on this device
    int num_sms = 0;
};

lora_status setup_current_device(DeviceSetup **out)
{
    static std::mutex mu;
    static DeviceSetup devices[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return LORA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return LORA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(mu);
    DeviceSetup &d = devices[dev];
    if (!d.ready) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return LORA_ERR_CUDA;
        if (major != 10 || minor != 3) return LORA_ERR_UNSUPPORTED;
        float *ptr = nullptr;
        if (cudaGetSymbolAddress((void **)&ptr, g_noalloc_scratch) != cudaSuccess || !ptr)
            return LORA_ERR_CUDA;
        d.scratch = ptr;
        d.num_sms = sms;
        d.ready = true;
    }
    *out = &d;
    return LORA_OK;
}

}  // namespace
}  // namespace lora

using namespace lora;

extern "C" lora_status lora_base_linear_noalloc(const void *X, const void *W_base, int T, int d_in,
                                                int d_out, void *Y, lora_stream_t stream)
{
    if (!X || !W_base || !Y || T < 0 || T > kDecodeMaxT) return LORA_ERR_ARG;
    if (d_in <= 0 || d_in > LORA_MAX_DIM || d_in % 8 || d_out <= 0 || d_out > LORA_MAX_DIM ||
        d_out % 8)
        return LORA_ERR_SHAPE;
    if (T == 0) return LORA_OK;
    DeviceSetup *dev = nullptr;
    lora_status st = setup_current_device(&dev);
    if (st != LORA_OK) return st;

    // fewer stream-K ranges when the partial sums would not fit the fixed scratch
    const size_t avail = kNoallocScratchFloats;
    const int no_pages = 0;
    DecodePlan plan;
    int max_G = dev->num_sms;
    for (;;) {
        if (!plan_decode(1, T, &d_in, &d_out, &no_pages, max_G, &plan)) return LORA_ERR_SHAPE;
        const size_t need = decode_partials_floats(plan);
        if (need <= avail) break;
        const size_t per_cta = (size_t)plan.max_seg * T * 128;
        const int fit = (int)(avail / per_cta);
        if (plan.G <= 1) return LORA_ERR_SHAPE;
        max_G = fit < plan.G ? (fit > 1 ? fit : 1) : plan.G - 1;
    }

    DecodeMaps maps;
    if (!make_tmap_bf16_2d(&maps.W[0], W_base, d_in, d_out, (uint64_t)d_in * 2, 64, 128) ||
        !make_tmap_bf16_2d(&maps.X[0], X, d_in, T, (uint64_t)d_in * 2, 64, plan.ntok))
        return LORA_ERR_ARG;
    // the partials need no clearing: every slot the finishing pass reads is
    // written by this call's GEMM kernel first
    int *err = nullptr;
    float *partials = dev->scratch;
    DecodeProblem &q = plan.prob[0];
    q.pool.d_in = d_in;
    q.pool.d_out = d_out;
    q.X = static_cast<const uint16_t *>(X);
    q.Y = static_cast<uint16_t *>(Y);
    q.err = err;
    cudaStream_t s = (cudaStream_t)stream;
    if (launch_gemm_decode(maps, plan, nullptr, partials, err, s) != cudaSuccess) return LORA_ERR_CUDA;
    if (launch_finish_decode(plan, partials, nullptr, s) != cudaSuccess) return LORA_ERR_CUDA;
    return LORA_OK;
}
