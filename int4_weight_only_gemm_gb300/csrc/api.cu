// C ABI of the W4A16 library: argument checks, per-M kernel choice,
// workspace bookkeeping and status reporting.  See include/w4a16.h.
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "dispatch_table.h"
#include "kernels.h"

namespace w4a16 {



namespace {

constexpr int kMaxDevices = 64;
std::atomic<uint64_t> g_launches{0};
std::mutex g_mu;
int g_sms[kMaxDevices];
void* g_ws[kMaxDevices];
size_t g_ws_bytes[kMaxDevices];

int current_device() {
    int d = -1;
    if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return -1;
    return d;
}

int device_sms(int dev) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_sms[dev] == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        g_sms[dev] = v;
    }
    return g_sms[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void* a, size_t an, const void* b, size_t bn) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + bn && b0 < a0 + an;
}

int check_kn(int N, int K) {
    if (N < 8 || K < 128 || N % 8 != 0) return W4A16_EINVAL;
    if (K % 128 != 0) return W4A16_EUNSUPPORTED;
    if ((long long)(K / 8) * N >= (1ll << 31)) return W4A16_EUNSUPPORTED;
    return W4A16_OK;
}

// Fused gate/up weights: H = columns of each half, a multiple of 64 so that
// every 128-column device tile holds 64 gate and 64 up columns.
int check_gate_up(int H, int K) {
    if (H < 64 || H % 64 != 0) return H < 1 ? W4A16_EINVAL : W4A16_EUNSUPPORTED;
    if (H > (1 << 29)) return W4A16_EUNSUPPORTED;
    return check_kn(2 * H, K);
}

int repack_gate_up(bool pack, const uint32_t* src, uint32_t* dst, int K, int H, cudaStream_t stream) {
    if (!src || !dst) return W4A16_EINVAL;
    int st = check_gate_up(H, K);
    if (st != W4A16_OK) return st;
    if (!aligned16(src) || !aligned16(dst)) return W4A16_EALIGN;
    const size_t bytes = (size_t)K / 2 * (2 * (size_t)H);
    if (overlaps(src, bytes, dst, bytes)) return W4A16_EINVAL;
    const cudaError_t e = pack ? launch_pack(src, dst, K, 2 * H, H, stream) : launch_unpack(src, dst, K, 2 * H, H, stream);
    if (e != cudaSuccess) return W4A16_ECUDA;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return W4A16_OK;
}

// The column-sliced GEMV gives every CTA whole columns: no split-K hand-off.
// Measured on the decoder's shapes and the vocabulary head at M = 1, 2, 4, 8
// it is as fast as the split-K form or faster (at M = 1: qkv 4.1 against
// 5.5 us, down 6.7 against 7.4, gate_up 8.2 against 8.2, vocabulary 46 against
// 49), provided its slices fill the GPU; with fewer columns than that the
// split-K form spreads K over the idle SMs.
bool gemv_uses_cs(int M, int N, int K, int sms, int guH, GemvCsPlan* cp) {
    return gemv_cs_plan(M, N, K, sms, guH, cp) && cp->ctas >= sms;
}

// Kernel choice for AUTO: the dispatch table's row (measured on GB300 over
// the decoder's shapes, see dispatch_table.h), provided the GEMV it names can
// run this problem; the tensor-core kernel otherwise.
int choose_path(int M, int N, int K, int sms) {
    const DispatchRow* r = dispatch_row(M, K, N);
    GemvPlan gp;
    GemvCsPlan cp;
    if (r && M <= 8) {
        if (r->path == W4A16_PATH_GEMV_CS && gemv_cs_plan(M, N, K, sms, 0, &cp)) return W4A16_PATH_GEMV_CS;
        if ((r->path == W4A16_PATH_GEMV_CS || r->path == W4A16_PATH_GEMV_SPLITK) && gemv_plan(M, N, K, sms, &gp))
            return W4A16_PATH_GEMV_SPLITK;
    }
    return W4A16_PATH_TC;
}

size_t ws_for_path(int path, int M, int N, int K, int sms) {
    GemvPlan gp;
    GemvCsPlan cp;
    if (path == W4A16_PATH_GEMV_CS) return 0;
    if (path == W4A16_PATH_GEMV) {
        // no workspace when both the plain and the fused gate/up product of
        // this N take the column-sliced form
        if (gemv_uses_cs(M, N, K, sms, 0, &cp) && gemv_uses_cs(M, N, K, sms, N / 2, &cp)) return 0;
        path = W4A16_PATH_GEMV_SPLITK;
    }
    if (path == W4A16_PATH_GEMV_SPLITK) return gemv_plan(M, N, K, sms, &gp) ? gp.ws_bytes : 0;
    TcPlan tp;
    return tc_plan(M, N, K, sms, &tp) ? tp.ws_bytes : 0;
}

// Launch flags used by the entry points that take none: programmatic dependent
// launch, which changes no ordering (every kernel waits for the preceding grid
// before it touches global memory) but lets its launch overlap that grid's end.
constexpr unsigned kDefaultFlags = W4A16_FLAG_PDL;
constexpr unsigned kKnownFlags = W4A16_FLAG_PDL | W4A16_FLAG_STATIC_WEIGHTS | W4A16_FLAG_TOKEN_TILE_MASK;

// guH > 0: fused gate/up weights with N = 2 guH columns, y = silu(gate) * up of [M][guH]
int run_gemm(int path, unsigned flags, const void* x, const uint32_t* qd, const void* scales, const uint32_t* qzeros,
             int M, int N, int K, int group, void* y, void* ws, size_t ws_bytes, cudaStream_t stream, int guH = 0) {
    if (flags & ~kKnownFlags) return W4A16_EINVAL;
    if (path < W4A16_PATH_AUTO || path > W4A16_PATH_GEMV_CS) return W4A16_EINVAL;
    int st = check_gemm(x, qd, scales, qzeros, M, N, K, group, y, guH ? guH : N);
    if (st != W4A16_OK || M == 0) return st;  // M == 0: nothing to compute
    const int dev = current_device();
    if (dev < 0) return W4A16_ECUDA;
    const int sms = device_sms(dev);
    if (sms <= 0) return W4A16_ECUDA;
    if (path == W4A16_PATH_AUTO) path = choose_path(M, N, K, sms);
    cudaError_t e;
    GemvCsPlan cp;
    if (path == W4A16_PATH_GEMV) path = gemv_uses_cs(M, N, K, sms, guH, &cp) ? W4A16_PATH_GEMV_CS : W4A16_PATH_GEMV_SPLITK;
    if (path == W4A16_PATH_GEMV_CS) {
        if (!gemv_cs_plan(M, N, K, sms, guH, &cp)) return W4A16_EUNSUPPORTED;
        e = launch_gemv_cs(static_cast<const uint16_t*>(x), qd, static_cast<const uint16_t*>(scales), qzeros,
                           static_cast<uint16_t*>(y), M, N, K, cp, stream, flags, guH);
    } else if (path == W4A16_PATH_GEMV_SPLITK) {
        GemvPlan gp;
        if (!gemv_plan(M, N, K, sms, &gp)) return W4A16_EUNSUPPORTED;
        if (gp.ws_bytes && (!ws || ws_bytes < gp.ws_bytes || !aligned16(ws))) return W4A16_EWORKSPACE;
        e = launch_gemv(static_cast<const uint16_t*>(x), qd, static_cast<const uint16_t*>(scales), qzeros,
                        static_cast<uint16_t*>(y), M, N, K, ws, gp, stream, flags, guH);
    } else if (path == W4A16_PATH_TC) {
        TcPlan tp;
        const int force_nt = (int)((flags & W4A16_FLAG_TOKEN_TILE_MASK) >> W4A16_FLAG_TOKEN_TILE_SHIFT);
        if (force_nt && force_nt != 16 && force_nt != 32 && force_nt != 64 && force_nt != 128 && force_nt != 192)
            return W4A16_EINVAL;
        if (!tc_plan(M, N, K, sms, &tp, force_nt)) return W4A16_EUNSUPPORTED;
        if (tp.ws_bytes && (!ws || ws_bytes < tp.ws_bytes || !aligned16(ws))) return W4A16_EWORKSPACE;
        e = launch_tc(static_cast<const uint16_t*>(x), qd, static_cast<const uint16_t*>(scales), qzeros,
                      static_cast<uint16_t*>(y), M, N, K, ws, tp, stream, flags, guH);
    } else {
        return W4A16_EINVAL;
    }
    if (e != cudaSuccess) return W4A16_ECUDA;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return W4A16_OK;
}

}  // namespace

// Argument rules of every GEMM entry point (also used by w4a16_gemm_noalloc).
// ny: columns of y (N for the plain product, N / 2 for the fused gate/up one)
int check_gemm(const void* x, const uint32_t* qd, const void* scales, const uint32_t* qzeros, int M, int N, int K,
               int group, void* y, int ny) {
    if (M < 0) return W4A16_EINVAL;
    if (M == 0) {  // an empty batch: only the shape is checked, no pointer is read
        if (group != 128) return W4A16_EUNSUPPORTED;
        return check_kn(N, K);
    }
    if (!x || !qd || !scales || !qzeros || !y) return W4A16_EINVAL;
    if (group != 128) return W4A16_EUNSUPPORTED;
    int st = check_kn(N, K);
    if (st != W4A16_OK) return st;
    if (!aligned16(x) || !aligned16(qd) || !aligned16(y) || !aligned16(scales) || !aligned16(qzeros))
        return W4A16_EALIGN;
    const size_t ybytes = (size_t)M * ny * 2;
    const int G = K / group;
    if (overlaps(y, ybytes, x, (size_t)M * K * 2) || overlaps(y, ybytes, qd, (size_t)K / 2 * N) ||
        overlaps(y, ybytes, scales, (size_t)G * N * 2) || overlaps(y, ybytes, qzeros, (size_t)G * N / 2))
        return W4A16_EINVAL;
    return W4A16_OK;
}

void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

const DispatchRow* dispatch_row(int M, int K, int N) {
    const long long kn = (long long)K * N;
    int cls = 0;
    while (cls < kDispatchClasses - 1 && kn > kClassMaxWeights[cls]) ++cls;
    const DispatchRow* last = nullptr;
    for (const DispatchRow& r : kDispatch) {
        if (r.cls != cls) continue;
        last = &r;
        if (M <= r.m_max) return &r;
    }
    return last;  // beyond the sweep: the largest M measured
}

int dispatch_nt(int M, int K, int N) {
    const DispatchRow* r = dispatch_row(M, K, N);
    return r && r->path == W4A16_PATH_TC ? r->nt : 0;
}

}  // namespace w4a16

using namespace w4a16;

extern "C" {

int w4a16_pack(const uint32_t* qweight, uint32_t* qweight_dev, int K, int N, w4a16_stream_t stream) {
    if (!qweight || !qweight_dev) return W4A16_EINVAL;
    int st = check_kn(N, K);
    if (st != W4A16_OK) return st;
    if (!aligned16(qweight) || !aligned16(qweight_dev)) return W4A16_EALIGN;
    const size_t bytes = (size_t)K / 2 * N;
    if (overlaps(qweight, bytes, qweight_dev, bytes)) return W4A16_EINVAL;
    if (launch_pack(qweight, qweight_dev, K, N, 0, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return W4A16_ECUDA;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return W4A16_OK;
}

int w4a16_unpack(const uint32_t* qweight_dev, uint32_t* qweight, int K, int N, w4a16_stream_t stream) {
    if (!qweight || !qweight_dev) return W4A16_EINVAL;
    int st = check_kn(N, K);
    if (st != W4A16_OK) return st;
    if (!aligned16(qweight) || !aligned16(qweight_dev)) return W4A16_EALIGN;
    const size_t bytes = (size_t)K / 2 * N;
    if (overlaps(qweight, bytes, qweight_dev, bytes)) return W4A16_EINVAL;
    if (launch_unpack(qweight_dev, qweight, K, N, 0, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return W4A16_ECUDA;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return W4A16_OK;
}

int w4a16_pack_gate_up(const uint32_t* qweight, uint32_t* qweight_dev, int K, int H, w4a16_stream_t stream) {
    return repack_gate_up(true, qweight, qweight_dev, K, H, reinterpret_cast<cudaStream_t>(stream));
}

int w4a16_unpack_gate_up(const uint32_t* qweight_dev, uint32_t* qweight, int K, int H, w4a16_stream_t stream) {
    return repack_gate_up(false, qweight_dev, qweight, K, H, reinterpret_cast<cudaStream_t>(stream));
}

int w4a16_gemm_gate_up_silu(int path, unsigned flags, const void* x, const uint32_t* qweight_dev, const void* scales,
                            const uint32_t* qzeros, int M, int H, int K, int group, void* y, void* workspace,
                            size_t workspace_bytes, w4a16_stream_t stream) {
    if (H < 1) return W4A16_EINVAL;
    const int st = check_gate_up(H, K);
    if (st != W4A16_OK) return st;
    return run_gemm(path, flags, x, qweight_dev, scales, qzeros, M, 2 * H, K, group, y, workspace, workspace_bytes,
                    reinterpret_cast<cudaStream_t>(stream), H);
}

int w4a16_requant_pack(const void* w, const void* scales, const uint32_t* qzeros, int K, int N, int group,
                       uint32_t* qweight_dev, w4a16_stream_t stream) {
    if (!w || !scales || !qzeros || !qweight_dev) return W4A16_EINVAL;
    if (group != 128) return W4A16_EUNSUPPORTED;
    int st = check_kn(N, K);
    if (st != W4A16_OK) return st;
    if (K / 128 * 4 > 65535) return W4A16_EUNSUPPORTED;  // one grid row per 32-row chunk
    if (!aligned16(w) || !aligned16(scales) || !aligned16(qzeros) || !aligned16(qweight_dev)) return W4A16_EALIGN;
    const size_t qbytes = (size_t)K / 2 * N;
    const int G = K / group;
    if (overlaps(qweight_dev, qbytes, w, (size_t)K * N * 2) || overlaps(qweight_dev, qbytes, scales, (size_t)G * N * 2) ||
        overlaps(qweight_dev, qbytes, qzeros, (size_t)G * N / 2))
        return W4A16_EINVAL;
    if (launch_requant_pack(static_cast<const uint16_t*>(w), static_cast<const uint16_t*>(scales), qzeros, qweight_dev,
                            K, N, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return W4A16_ECUDA;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return W4A16_OK;
}

size_t w4a16_workspace_bytes_path(int path, int M, int N, int K, int group) {
    if (M < 1 || group != 128 || check_kn(N, K) != W4A16_OK) return 0;
    const int dev = current_device();
    if (dev < 0) return 0;
    const int sms = device_sms(dev);
    if (sms <= 0) return 0;
    if (path == W4A16_PATH_AUTO) path = choose_path(M, N, K, sms);
    return ws_for_path(path, M, N, K, sms);
}

size_t w4a16_workspace_bytes(int M, int N, int K, int group) {
    return w4a16_workspace_bytes_path(W4A16_PATH_AUTO, M, N, K, group);
}

size_t w4a16_workspace_bytes_max(int max_M, int N, int K, int group) {
    size_t best = 0;
    for (int m = 1; m <= max_M; ++m) {
        // the plan only changes at token-tile boundaries; probe each M up to 256, then tile edges
        if (m > 256 && (m % 128) != 0 && m != max_M) continue;
        for (int path = W4A16_PATH_GEMV; path <= W4A16_PATH_GEMV_CS; ++path) {
            size_t b = w4a16_workspace_bytes_path(path, m, N, K, group);
            if (b > best) best = b;
        }
        // every token tile the tuning flag can force
        const int dev = current_device();
        const int sms = dev >= 0 ? device_sms(dev) : 0;
        if (sms > 0 && group == 128 && check_kn(N, K) == W4A16_OK) {
            for (int nt : {16, 32, 64, 128, 192}) {
                TcPlan tp;
                if (tc_plan(m, N, K, sms, &tp, nt) && tp.ws_bytes > best) best = tp.ws_bytes;
            }
        }
    }
    return best;
}

int w4a16_set_workspace(void* workspace, size_t bytes) {
    const int dev = current_device();
    if (dev < 0) return W4A16_ECUDA;
    if (workspace && !aligned16(workspace)) return W4A16_EALIGN;
    std::lock_guard<std::mutex> lk(g_mu);
    g_ws[dev] = workspace;
    g_ws_bytes[dev] = workspace ? bytes : 0;
    return W4A16_OK;
}

int w4a16_gemm_path(int path, const void* x, const uint32_t* qweight_dev, const void* scales, const uint32_t* qzeros,
                    int M, int N, int K, int group, void* y, void* workspace, size_t workspace_bytes,
                    w4a16_stream_t stream) {
    return run_gemm(path, kDefaultFlags, x, qweight_dev, scales, qzeros, M, N, K, group, y, workspace,
                    workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

int w4a16_gemm_ex(int path, unsigned flags, const void* x, const uint32_t* qweight_dev, const void* scales,
                  const uint32_t* qzeros, int M, int N, int K, int group, void* y, void* workspace,
                  size_t workspace_bytes, w4a16_stream_t stream) {
    return run_gemm(path, flags, x, qweight_dev, scales, qzeros, M, N, K, group, y, workspace, workspace_bytes,
                    reinterpret_cast<cudaStream_t>(stream));
}

int w4a16_gemm_ws(const void* x, const uint32_t* qweight_dev, const void* scales, const uint32_t* qzeros, int M,
                  int N, int K, int group, void* y, void* workspace, size_t workspace_bytes, w4a16_stream_t stream) {
    return run_gemm(W4A16_PATH_AUTO, kDefaultFlags, x, qweight_dev, scales, qzeros, M, N, K, group, y, workspace,
                    workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

int w4a16_gemm(const void* x, const uint32_t* qweight_dev, const void* scales, const uint32_t* qzeros, int M, int N,
               int K, int group, void* y, w4a16_stream_t stream) {
    const int dev = current_device();
    if (dev < 0) return W4A16_ECUDA;
    void* ws;
    size_t wsb;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        ws = g_ws[dev];
        wsb = g_ws_bytes[dev];
    }
    return run_gemm(W4A16_PATH_AUTO, kDefaultFlags, x, qweight_dev, scales, qzeros, M, N, K, group, y, ws, wsb,
                    reinterpret_cast<cudaStream_t>(stream));
}

int w4a16_auto_path(int M, int N, int K, int group) {
    if (M < 1 || group != 128 || check_kn(N, K) != W4A16_OK) return W4A16_EINVAL;
    const int dev = current_device();
    if (dev < 0) return W4A16_ECUDA;
    const int sms = device_sms(dev);
    if (sms <= 0) return W4A16_ECUDA;
    return choose_path(M, N, K, sms);
}

const char* w4a16_status_str(int status) {
    switch (status) {
        case W4A16_OK: return "ok";
        case W4A16_EINVAL: return "invalid argument (null pointer, bad size or overlapping output)";
        case W4A16_EALIGN: return "pointer not 16-byte aligned";
        case W4A16_EUNSUPPORTED: return "unsupported problem (group must be 128, K a multiple of 128)";
        case W4A16_ECUDA: return "CUDA runtime error or failed launch";
        case W4A16_ETIMEOUT: return "a bounded device-side wait timed out";
        case W4A16_EWORKSPACE: return "workspace missing, too small or misaligned";
        default: return "unknown status";
    }
}

int w4a16_last_device_status(w4a16_stream_t stream) {
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return W4A16_ECUDA;
    const int a = gemv_read_status();
    const int b = tc_read_status();
    const int c = selftest_read_status();
    const int d = swa_read_status();
    if (a == W4A16_ECUDA || b == W4A16_ECUDA || c == W4A16_ECUDA || d == W4A16_ECUDA) return W4A16_ECUDA;
    if (a != 0) return a;
    if (b != 0) return b;
    if (d != 0) return d;
    return c;
}

int w4a16_selftest_wait_timeout(long long wait_ns, w4a16_stream_t stream) {
    if (wait_ns < 1000 || wait_ns > 1000000000ll) return W4A16_EINVAL;
    if (launch_selftest_wait((uint64_t)wait_ns, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return W4A16_ECUDA;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return W4A16_OK;
}

static int check_swa(int nq, int Hq, int Hkv, int head_dim, int L, int Lmax, int window, int block) {
    if (nq < 1 || Hq < 1 || Hkv < 1 || L < nq || Lmax < L || window < 1 || (block != 0 && block != 1))
        return W4A16_EINVAL;
    if (Hq % Hkv != 0 || Lmax % 8 != 0) return W4A16_EINVAL;
    if (head_dim != 128) return W4A16_EUNSUPPORTED;
    if ((long long)nq * (Hq / Hkv) > 128 || Hkv > 65535) return W4A16_EUNSUPPORTED;
    return W4A16_OK;
}

size_t w4a16_swa_workspace_bytes(int nq, int Hq, int Hkv, int head_dim, int L, int window, int block) {
    if (check_swa(nq, Hq, Hkv, head_dim, L, (L + 7) & ~7, window, block) != W4A16_OK) return 0;
    SwaPlan sp;
    if (!swa_plan(nq, Hq, Hkv, L, window, block, &sp)) return 0;
    return sp.ws_bytes;
}

int w4a16_swa_attention(const void* q, const void* k_cache, const void* vt_cache, int nq, int Hq, int Hkv,
                        int head_dim, int L, int Lmax, int window, int block, void* out, void* workspace,
                        size_t workspace_bytes, unsigned flags, w4a16_stream_t stream) {
    if (!q || !k_cache || !vt_cache || !out) return W4A16_EINVAL;
    if (flags & ~(unsigned)W4A16_FLAG_PDL) return W4A16_EINVAL;
    int st = check_swa(nq, Hq, Hkv, head_dim, L, Lmax, window, block);
    if (st != W4A16_OK) return st;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(vt_cache) || !aligned16(out)) return W4A16_EALIGN;
    const size_t qbytes = (size_t)nq * Hq * head_dim * 2;
    const size_t cbytes = (size_t)Hkv * Lmax * head_dim * 2;
    if (overlaps(out, qbytes, q, qbytes) || overlaps(out, qbytes, k_cache, cbytes) ||
        overlaps(out, qbytes, vt_cache, cbytes))
        return W4A16_EINVAL;
    SwaPlan sp;
    if (!swa_plan(nq, Hq, Hkv, L, window, block, &sp)) return W4A16_EUNSUPPORTED;
    if (!workspace || workspace_bytes < sp.ws_bytes || !aligned16(workspace)) return W4A16_EWORKSPACE;
    if (launch_swa(static_cast<const uint16_t*>(q), static_cast<const uint16_t*>(k_cache),
                   static_cast<const uint16_t*>(vt_cache), static_cast<uint16_t*>(out), nq, Hq, Hkv, L, Lmax, window,
                   block, workspace, sp, reinterpret_cast<cudaStream_t>(stream), (flags & W4A16_FLAG_PDL) != 0) !=
        cudaSuccess)
        return W4A16_ECUDA;
    g_launches.fetch_add(2, std::memory_order_relaxed);  // the chunk kernel and the combine
    return W4A16_OK;
}

uint64_t w4a16_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
