// Split-K GEMV for M = 1..8 on CUDA cores (sm_103a).
//
// y[m][n] = sum_k x[m][k] (q[k][n] - z[g][n]) s[g][n], g = k / 128: the INT4
// linear layer run at every decode step by the quantized target and drafter
// of "Quantize the Target, Quantize the Drafter" (pith.science review,
// referee report summary; group size 128 from "Assumptions & free
// parameters").
//
// Work split (stream-K): the packed weights are a sequence of C chunks of
// 32 rows x one 128-column tile (2 KB, contiguous in the device layout, in
// (tile, K) order).  P workers (128-thread warpgroups, 4 per CTA, one CTA per
// SM) take contiguous chunk ranges of equal length, so every SM streams the
// same number of bytes.  Thread t of a worker owns column t of the current
// tile and reads its 4 words of a chunk with one 128-bit load; a warp's load
// is 512 contiguous bytes.
//
// Arithmetic per chunk and token: dot = sum_k (128 + q_k) x_k, with the
// bfloat16 value 128 + q made by one mask-and-or per pair of rows (exact), and
// bf16 x bf16 -> f32 fused multiply-adds; then the zero point and scale are
// applied once per chunk in f32: acc += s (dot - (128 + z) sum_k x_k), using a
// per-chunk activation sum computed once per CTA.  The scale is used at its
// full binary16 precision.
//
// Partial tiles (a worker range that starts or ends inside a tile) go to the
// workspace; the last worker to arrive on a tile (per-tile counter) adds the
// partials in worker order -- deterministic -- and writes y.
#include "common.cuh"
#include "kernels.h"

namespace w4a16 {

static __device__ int g_gemv_status;

struct GemvParams {
    const uint16_t* x;
    const uint32_t* qd;
    const uint16_t* scales;
    const uint32_t* qzeros;
    uint16_t* y;
    uint32_t* counters;
    float* partials;
    int M, N, K, KB, NB;
    int cpt;        // chunks per tile = 4 * KB
    long long C;    // total chunks
    int P;          // workers
    int prefetch;   // weights may be loaded before the preceding grid completes
};

constexpr int kGemvWG = 4;  // worker warpgroups per CTA
constexpr int kGemvMaxSmem = 200 * 1024;  // activation copy + chunk sums

__device__ __forceinline__ long long worker_begin(long long w, long long C, int P) { return w * C / P; }
__device__ __forceinline__ int worker_of(long long c, long long C, int P) {
    return (int)(((c + 1) * (long long)P - 1) / C);
}

__device__ __forceinline__ uint4 ld_stream_v4(const uint32_t* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void wg_bar(int wg) {
    asm volatile("bar.sync %0, 128;" ::"r"(wg + 1) : "memory");
}

template <int M>
__device__ __forceinline__ void gemv_flush(const GemvParams& p, int worker, int wg, int t, int nb, long long a,
                                           long long b, long long my_begin, float (&acc)[M], int* sh_last) {
    const Layout L(p.K, p.N);
    const int W = L.width(nb);
    const int n = 128 * nb + t;
    const long long t0 = (long long)nb * p.cpt, t1 = t0 + p.cpt;
    if (a == t0 && b == t1) {  // whole tile owned: write y directly
        if (t < W) {
#pragma unroll
            for (int m = 0; m < M; ++m)
                if (m < p.M) p.y[(size_t)m * p.N + n] = f32_to_bf16_rn(acc[m]);
        }
        return;
    }
    const int slot = (my_begin / p.cpt == nb) ? 0 : 1;
    float* part = p.partials + ((size_t)(worker * 2 + slot) * M) * 128;
#pragma unroll
    for (int m = 0; m < M; ++m) part[m * 128 + t] = acc[m];
    __threadfence();
    wg_bar(wg);
    if (t == 0) {
        const int wf = worker_of(t0, p.C, p.P), wl = worker_of(t1 - 1, p.C, p.P);
        const unsigned target = (unsigned)(wl - wf + 1);
        const unsigned old = atomicAdd(&p.counters[nb], 1u);
        sh_last[wg] = (old == target - 1) ? 1 : 0;
    }
    wg_bar(wg);
    if (sh_last[wg]) {
        __threadfence();
        const int wf = worker_of(t0, p.C, p.P), wl = worker_of(t1 - 1, p.C, p.P);
        float sum[M];
#pragma unroll
        for (int m = 0; m < M; ++m) sum[m] = 0.f;
        for (int w = wf; w <= wl; ++w) {
            const int s = (worker_begin(w, p.C, p.P) / p.cpt == nb) ? 0 : 1;
            const float* q = p.partials + ((size_t)(w * 2 + s) * M) * 128;
#pragma unroll
            for (int m = 0; m < M; ++m) sum[m] += __ldcg(q + m * 128 + t);
        }
        if (t < W) {
#pragma unroll
            for (int m = 0; m < M; ++m)
                if (m < p.M) p.y[(size_t)m * p.N + n] = f32_to_bf16_rn(sum[m]);
        }
        if (t == 0) p.counters[nb] = 0u;
    }
}

template <int M, int D>
__global__ void __launch_bounds__(128 * kGemvWG, 1) gemv_kernel(const GemvParams p) {
    extern __shared__ __align__(16) unsigned char smem[];
    uint16_t* xs = reinterpret_cast<uint16_t*>(smem);                           // [M][K] bf16
    float* xsum = reinterpret_cast<float*>(smem + (size_t)M * p.K * 2);         // [M][K/32]
    __shared__ int sh_last[kGemvWG];

    const int tid = threadIdx.x;
    const int wg = tid >> 7;
    const int t = tid & 127;
    const int worker = blockIdx.x * kGemvWG + wg;
    const Layout L(p.K, p.N);
    const long long c_begin = worker < p.P ? worker_begin(worker, p.C, p.P) : 0;
    const long long c_end = worker < p.P ? worker_begin(worker + 1, p.C, p.P) : 0;

    // 1. first weight loads go out before anything else
    uint4 buf[D];
    auto load_chunk = [&](long long c) -> uint4 {
        const int nb = (int)(c / p.cpt);
        const int rem = (int)(c - (long long)nb * p.cpt);
        const int W = L.width(nb);
        if (t >= W) return make_uint4(0, 0, 0, 0);
        const uint32_t* src = p.qd + L.block_word(nb, rem >> 2) + ((size_t)(rem & 3) * W + t) * 4;
        return ld_stream_v4(src);
    };
    // With static weights the first loads go out before waiting on the
    // preceding grid; otherwise after it (x, y and the workspace are always
    // touched only after the wait).
    if (p.prefetch) {
#pragma unroll
        for (int i = 0; i < D; ++i) buf[i] = (c_begin + i < c_end) ? load_chunk(c_begin + i) : make_uint4(0, 0, 0, 0);
    }
    pdl_wait();
    if (!p.prefetch) {
#pragma unroll
        for (int i = 0; i < D; ++i) buf[i] = (c_begin + i < c_end) ? load_chunk(c_begin + i) : make_uint4(0, 0, 0, 0);
    }
    pdl_launch_dependents();  // one wave: the next grid can only start where this one ends

    // 2. activations to shared memory, then per-chunk sums
    {
        const int nvec = p.M * p.K / 8;  // 16-byte vectors of x actually present
        const uint4* xg = reinterpret_cast<const uint4*>(p.x);
        uint4* xv = reinterpret_cast<uint4*>(xs);
        for (int i = tid; i < M * p.K / 8; i += blockDim.x) xv[i] = i < nvec ? __ldg(xg + i) : make_uint4(0, 0, 0, 0);
        __syncthreads();
        const int nk = p.K / 32;
        for (int i = tid; i < M * nk; i += blockDim.x) {
            const uint32_t* xr = reinterpret_cast<const uint32_t*>(xs) + (size_t)i * 16;  // 32 bf16
            float s = 0.f;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const uint32_t v = xr[e];
                s += bf16lo(v);
                s += bf16hi(v);
            }
            xsum[i] = s;
        }
        __syncthreads();
    }
    if (worker >= p.P) return;  // no named barrier is shared across warpgroups

    float acc[M];
#pragma unroll
    for (int m = 0; m < M; ++m) acc[m] = 0.f;
    int cur_nb = (int)(c_begin / p.cpt);
    long long seg_first = c_begin;

    for (long long c0 = c_begin; c0 < c_end; c0 += D) {
#pragma unroll
        for (int i = 0; i < D; ++i) {
            const long long c = c0 + i;
            if (c < c_end) {
                const uint4 cur = buf[i];
                if (c + D < c_end) buf[i] = load_chunk(c + D);
                const int nb = (int)(c / p.cpt);
                if (nb != cur_nb) {
                    gemv_flush<M>(p, worker, wg, t, cur_nb, seg_first, c, c_begin, acc, sh_last);
#pragma unroll
                    for (int m = 0; m < M; ++m) acc[m] = 0.f;
                    cur_nb = nb;
                    seg_first = c;
                }
                const int rem = (int)(c - (long long)nb * p.cpt);
                const int kb = rem >> 2;
                const int k0 = kb * 128 + (rem & 3) * 32;
                const int n = 128 * nb + t;
                if (t < L.width(nb)) {
                    const float s = f16_bits_to_f32(__ldg(p.scales + (size_t)kb * p.N + n));
                    const uint32_t zw = __ldg(p.qzeros + (size_t)kb * (p.N / 8) + (n >> 3));
                    const float zoff = 128.f + (float)((zw >> (4 * (n & 7))) & 0xFu);
                    // four independent accumulation chains per token (one per word)
                    float d[4][M];
                    const uint32_t wv[4] = {cur.x, cur.y, cur.z, cur.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint32_t wp[4];
#pragma unroll
                        for (int q = 0; q < 4; ++q) wp[q] = magic_pair(wv[j], q);
#pragma unroll
                        for (int m = 0; m < M; ++m) {
                            const uint4 xq = *reinterpret_cast<const uint4*>(xs + (size_t)m * p.K + k0 + 8 * j);
                            const uint32_t xp[4] = {xq.x, xq.y, xq.z, xq.w};
                            float a = 0.f;
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                a = fma_lo(wp[q], xp[q], a);
                                a = fma_hi(wp[q], xp[q], a);
                            }
                            d[j][m] = a;
                        }
                    }
                    const int kc = k0 >> 5;
#pragma unroll
                    for (int m = 0; m < M; ++m) {
                        const float dot = (d[0][m] + d[1][m]) + (d[2][m] + d[3][m]);
                        acc[m] = fmaf(s, fmaf(-zoff, xsum[m * (p.K / 32) + kc], dot), acc[m]);
                    }
                }
            }
        }
    }
    gemv_flush<M>(p, worker, wg, t, cur_nb, seg_first, c_end, c_begin, acc, sh_last);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------


static int gemv_mtile(int M) { return M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : 8; }

bool gemv_plan(int M, int N, int K, int sms, GemvPlan* out) {
    if (M < 1 || M > 8) return false;
    const int MT = gemv_mtile(M);
    const Layout L(K, N);
    const long long C = (long long)L.NB * 4 * L.KB;
    const size_t smem = (size_t)MT * K * 2 + (size_t)MT * (K / 32) * 4;
    if (smem > (size_t)kGemvMaxSmem) return false;
    if ((size_t)L.NB > kMaxCounters) return false;
    long long P = (long long)sms * kGemvWG;
    if (P > C) P = C;
    const int ctas = (int)((P + kGemvWG - 1) / kGemvWG);
    out->ctas = ctas;
    out->P = (int)P;
    out->C = C;
    out->smem = smem;
    out->ws_bytes = ws_counter_bytes(L.NB) + (size_t)P * 2 * MT * 128 * sizeof(float);
    return true;
}

template <int M>
static cudaError_t launch_m(const GemvParams& prm, const GemvPlan& plan, cudaStream_t s, bool pdl) {
    constexpr int D = 4;
    auto kern = gemv_kernel<M, D>;
    // the dynamic shared memory limit is raised once per device to the maximum
    // any plan asks for, so that launches (also inside graph capture) make no
    // other runtime calls
    static int set_for[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!set_for[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemvMaxSmem);
        if (e != cudaSuccess) return e;
        set_for[dev] = 1;
    }
    return launch_kernel(kern, dim3(plan.ctas), dim3(128 * kGemvWG), plan.smem, s, pdl, prm);
}

cudaError_t launch_gemv(const uint16_t* x, const uint32_t* qd, const uint16_t* scales, const uint32_t* qzeros,
                        uint16_t* y, int M, int N, int K, void* ws, const GemvPlan& plan, cudaStream_t s,
                        unsigned flags) {
    const Layout L(K, N);
    GemvParams prm;
    prm.x = x;
    prm.qd = qd;
    prm.scales = scales;
    prm.qzeros = qzeros;
    prm.y = y;
    prm.counters = reinterpret_cast<uint32_t*>(ws);
    prm.partials = reinterpret_cast<float*>(reinterpret_cast<char*>(ws) + ws_counter_bytes(L.NB));
    prm.M = M;
    prm.N = N;
    prm.K = K;
    prm.KB = L.KB;
    prm.NB = L.NB;
    prm.cpt = 4 * L.KB;
    prm.C = plan.C;
    prm.P = plan.P;
    const bool pdl = (flags & W4A16_FLAG_PDL) != 0;
    prm.prefetch = pdl && (flags & W4A16_FLAG_STATIC_WEIGHTS) ? 1 : 0;
    switch (gemv_mtile(M)) {
        case 1: return launch_m<1>(prm, plan, s, pdl);
        case 2: return launch_m<2>(prm, plan, s, pdl);
        case 4: return launch_m<4>(prm, plan, s, pdl);
        default: return launch_m<8>(prm, plan, s, pdl);
    }
}

int gemv_read_status() {
    int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_gemv_status, sizeof(int)) != cudaSuccess) return W4A16_ECUDA;
    if (cudaMemcpyToSymbol(g_gemv_status, &zero, sizeof(int)) != cudaSuccess) return W4A16_ECUDA;
    return v;
}

}  // namespace w4a16
