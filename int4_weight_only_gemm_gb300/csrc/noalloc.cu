// w4a16_gemm_noalloc: the split-K GEMV (M <= 8) with its scratch memory held
// by the library itself, for callers that cannot allocate device memory.
//
// Who needs it: code that is handed only its inputs and outputs and may not
// allocate -- a plugin inside an inference runtime that owns and plans all
// device memory, a process whose allocator is locked down or budgeted to the
// byte, a host routine that must not risk an allocation failure or the
// device-wide synchronisation cudaMalloc can cause.  The regular entry points
// need a caller-provided workspace for their split-K partial sums; this one
// uses a fixed array compiled into the library instead.
//
// The array lives in every GPU that loads the library until the process
// exits.  All calls on a device share it, so calls that may overlap on the GPU
// (different streams, or different host threads) race and must be serialised
// by the caller.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace w4a16 {
namespace {

// Split-K scratch: arrival counters (first 64 KB) and partial sums.
constexpr size_t kNoAllocScratch = W4A16_NOALLOC_SCRATCH_BYTES;
static_assert(kNoAllocScratch > kCounterBytes, "scratch must hold the counter area");
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratch];

constexpr int kMaxDev = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDev];  // device address of g_noalloc_scratch, per device
int g_noalloc_sms[kMaxDev];

// Once per device, with that device current: the host name of the array is
// only a stand-in, so its device address is looked up and kept.
int setup_device(int dev, void** ptr, int* sms) {
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return W4A16_ECUDA;
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
            return W4A16_ECUDA;
        g_noalloc_sms[dev] = v;
        g_noalloc_ptr[dev] = p;
    }
    *ptr = g_noalloc_ptr[dev];
    *sms = g_noalloc_sms[dev];
    return W4A16_OK;
}

}  // namespace
}  // namespace w4a16

using namespace w4a16;

extern "C" int w4a16_gemm_noalloc(const void* x, const uint32_t* qweight_dev, const void* scales,
                                  const uint32_t* qzeros, int M, int N, int K, int group, void* y,
                                  w4a16_stream_t stream) {
    // the same argument rules as w4a16_gemm
    const int chk = check_gemm(x, qweight_dev, scales, qzeros, M, N, K, group, y, N);
    if (chk != W4A16_OK || M == 0) return chk;  // M == 0: nothing to compute
    if (M > 8) return W4A16_EUNSUPPORTED;  // only the GEMV has a no-allocation form

    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return W4A16_ECUDA;
    void* scratch = nullptr;
    int sms = 0;
    const int st = setup_device(dev, &scratch, &sms);
    if (st != W4A16_OK) return st;

    GemvPlan plan;
    if (!gemv_plan(M, N, K, sms, &plan)) return W4A16_EUNSUPPORTED;
    // The GEMV's scratch is 64 KB of counters plus one 128 x MT block of f32
    // partials per CTA (MT <= 8): at most 64 KB + CTAs * 4 KB, about 0.7 MB on
    // a 152-SM GPU, well inside the array.  The check guards against a plan
    // that would ever need more.
    if (plan.ws_bytes > kNoAllocScratch) return W4A16_EWORKSPACE;

    // The arrival counters must start at zero; the array keeps whatever the
    // last call left, so the ones this problem uses are cleared first.
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const size_t ntiles = (size_t)(N + 127) / 128;
    if (cudaMemsetAsync(scratch, 0, ntiles * sizeof(uint32_t), s) != cudaSuccess) return W4A16_ECUDA;
    if (launch_gemv(static_cast<const uint16_t*>(x), qweight_dev, static_cast<const uint16_t*>(scales), qzeros,
                    static_cast<uint16_t*>(y), M, N, K, scratch, plan, s, 0u, 0) != cudaSuccess)
        return W4A16_ECUDA;
    note_launch();
    return W4A16_OK;
}
