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
    int C;          // total chunks
    int P;          // workers
    int q, r;       // C = q * P + r: worker w takes q chunks, plus one if w < r
    int prefetch;   // weights may be loaded before the preceding grid completes
};

constexpr int kGemvWG = 4;  // worker warpgroups per CTA
constexpr int kGemvMaxSmem = 200 * 1024;  // activation copy + chunk sums

// Division-free equal split of the C chunks over P workers.
__device__ __forceinline__ int worker_begin(int w, const GemvParams& p) { return w * p.q + (w < p.r ? w : p.r); }
__device__ __forceinline__ int worker_of(int c, const GemvParams& p) {
    const int big = p.r * (p.q + 1);
    return c < big ? c / (p.q + 1) : p.r + (c - big) / p.q;
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

// One chunk's data for one thread: its column's 4 words (32 rows), the
// group's scale (binary16 bits) and the word holding its zero point.
struct ChunkData {
    uint4 w;
    uint32_t s, zw;
};

// Write a finished tile segment: directly when this worker owns the whole
// tile, else as a partial sum with the ordered last-arrival reduction.
template <int M>
__device__ __forceinline__ void gemv_flush(const GemvParams& p, int worker, int wg, int t, int nb, int a, int b,
                                           int my_begin, const float (&acc)[M], int* sh_last) {
    const Layout L(p.K, p.N);
    const int W = L.width(nb);
    const int n = 128 * nb + t;
    const int t0 = nb * p.cpt, t1 = t0 + p.cpt;
    if (a == t0 && b == t1) {
        if (t < W) {
#pragma unroll
            for (int m = 0; m < M; ++m)
                if (m < p.M) p.y[(size_t)m * p.N + n] = f32_to_bf16_rn(acc[m]);
        }
        return;
    }
    const int slot = (my_begin >= t0) ? 0 : 1;  // first tile of this worker, or its last
    float* part = p.partials + ((size_t)(worker * 2 + slot) * M) * 128;
#pragma unroll
    for (int m = 0; m < M; ++m) part[m * 128 + t] = acc[m];
    __threadfence();
    wg_bar(wg);
    const int wf = worker_of(t0, p), wl = worker_of(t1 - 1, p);
    if (t == 0) {
        const unsigned old = atomicAdd(&p.counters[nb], 1u);
        sh_last[wg] = (old == (unsigned)(wl - wf)) ? 1 : 0;
    }
    wg_bar(wg);
    if (sh_last[wg]) {
        __threadfence();
        float sum[M];
#pragma unroll
        for (int m = 0; m < M; ++m) sum[m] = 0.f;
        for (int w = wf; w <= wl; ++w) {  // fixed order: deterministic
            const int s = (worker_begin(w, p) >= t0) ? 0 : 1;
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
    const bool active = worker < p.P;
    const int c_begin = active ? worker_begin(worker, p) : 0;
    const int c_end = active ? worker_begin(worker + 1, p) : 0;

    // Load cursor: chunks are fetched in increasing order, D ahead of use,
    // through pointers that advance by constant steps.  In full tiles chunk
    // c sits at word 512 c; in the ragged last tile chunks are W*4 words.
    // Threads beyond a ragged tile's width read column W-1 (a valid address)
    // and discard the result, so the loop has no per-thread branches.
    int l_nb = c_begin / (p.cpt > 0 ? p.cpt : 1);
    int l_rem = c_begin - l_nb * p.cpt;
    int l_left = c_end - c_begin;
    const uint32_t* wp;
    const uint16_t* sp;
    const uint32_t* zp;
    int wstep;
    auto seek_tile = [&]() {  // pointers for chunk (l_nb, l_rem)
        const int W = L.width(l_nb);
        const int tc = t < W ? t : W - 1;
        const int kb = l_rem >> 2;
        wstep = W * 4;  // one chunk: W columns x 4 words
        wp = p.qd + L.block_word(l_nb, kb) + ((size_t)(l_rem & 3) * W + tc) * 4;
        const int n = 128 * l_nb + tc;
        sp = p.scales + (size_t)kb * p.N + n;
        zp = p.qzeros + (size_t)kb * (p.N / 8) + (n >> 3);
    };
    if (l_left > 0) seek_tile();
    else {
        wp = p.qd;
        sp = p.scales;
        zp = p.qzeros;
        wstep = 0;
    }
    auto next_chunk = [&]() -> ChunkData {
        ChunkData d;
        d.w = ld_stream_v4(wp);
        d.s = __ldg(sp);
        d.zw = __ldg(zp);
        if (l_left > 1) {
            --l_left;
            ++l_rem;
            if (l_rem == p.cpt) {  // next tile (rare, uniform across the warpgroup)
                l_rem = 0;
                ++l_nb;
                seek_tile();
            } else {
                wp += wstep;
                if ((l_rem & 3) == 0) {  // next group of 128 rows
                    sp += p.N;
                    zp += p.N / 8;
                }
            }
        } else {
            l_left = 0;  // stay on the last chunk: later loads re-read it and are never used
        }
        return d;
    };

    // With static weights the first loads go out before waiting on the
    // preceding grid; otherwise after it (x, y and the workspace are always
    // touched only after the wait).
    ChunkData buf[D];
    if (p.prefetch) {
#pragma unroll
        for (int i = 0; i < D; ++i) buf[i] = next_chunk();
    }
    pdl_wait();
    if (!p.prefetch) {
#pragma unroll
        for (int i = 0; i < D; ++i) buf[i] = next_chunk();
    }
    pdl_launch_dependents();  // one wave: the next grid can only start where this one ends

    // activations to shared memory, then per-32-row chunk sums
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
    if (!active) return;  // no named barrier is shared across warpgroups

    // Tile segments: [seg_a, seg_b) lies in one tile.  Buffer slot i holds
    // chunk c with (c - c_begin) % D == i, so segments walk the same D-groups.
    int seg_a = c_begin;
    int group_base = c_begin;
    while (seg_a < c_end) {
        const int nb = seg_a / p.cpt;
        const int tile_end = (nb + 1) * p.cpt;
        const int seg_b = c_end < tile_end ? c_end : tile_end;
        const int n = 128 * nb + t;
        const int zshift = 4 * (n & 7);
        float acc[M];
#pragma unroll
        for (int m = 0; m < M; ++m) acc[m] = 0.f;
        for (int base = group_base; base < seg_b; base += D) {
#pragma unroll
            for (int i = 0; i < D; ++i) {
                const int c = base + i;
                if (c >= seg_a && c < seg_b) {
                    const ChunkData cur = buf[i];
                    buf[i] = next_chunk();
                    {
                        const int rem = c - nb * p.cpt;
                        const int k0 = (rem >> 2) * 128 + (rem & 3) * 32;
                        const float s = f16_bits_to_f32((uint16_t)cur.s);
                        const float zoff = 128.f + (float)((cur.zw >> zshift) & 0xFu);
                        // four independent accumulation chains per token (one per word)
                        float d[4][M];
                        const uint32_t wv[4] = {cur.w.x, cur.w.y, cur.w.z, cur.w.w};
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            uint32_t wp[4];
#pragma unroll
                            for (int qq = 0; qq < 4; ++qq) wp[qq] = magic_pair(wv[j], qq);
#pragma unroll
                            for (int m = 0; m < M; ++m) {
                                const uint4 xq = *reinterpret_cast<const uint4*>(xs + (size_t)m * p.K + k0 + 8 * j);
                                const uint32_t xp[4] = {xq.x, xq.y, xq.z, xq.w};
                                float a = 0.f;
#pragma unroll
                                for (int qq = 0; qq < 4; ++qq) {
                                    a = fma_lo(wp[qq], xp[qq], a);
                                    a = fma_hi(wp[qq], xp[qq], a);
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
        gemv_flush<M>(p, worker, wg, t, nb, seg_a, seg_b, c_begin, acc, sh_last);
        group_base = seg_b - (seg_b - c_begin) % D;
        seg_a = seg_b;
    }
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
    if (C >= (1ll << 31)) return false;
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
    constexpr int D = M == 1 ? 8 : M == 2 ? 6 : M == 4 ? 4 : 2;  // chunks in flight per thread
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
    prm.C = (int)plan.C;
    prm.P = plan.P;
    prm.q = (int)(plan.C / plan.P);
    prm.r = (int)(plan.C % plan.P);
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
