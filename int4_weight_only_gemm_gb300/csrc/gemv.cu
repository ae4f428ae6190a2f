// Split-K GEMV for M = 1..8 on CUDA cores (sm_103a).
//
// y[m][n] = sum_k x[m][k] (q[k][n] - z[g][n]) s[g][n], g = k / 128: the INT4
// linear layer run at every decode step by the quantized target and drafter
// of "Quantize the Target, Quantize the Drafter" (pith.science review,
// referee report summary; group size 128 from "Assumptions & free
// parameters").
//
// Work split: a unit is one 128-row group of K of one 128-column tile (8 KB
// of packed weights, contiguous in the device layout), units in (tile, K)
// order, one CTA per SM.  With at least as many tiles as CTAs, each CTA takes
// a range of whole tiles.  With fewer, each tile is cut into P/T pieces
// (rounded down or up, P CTAs, T tiles) of contiguous units, one CTA per
// piece: every CTA then streams about the same number of bytes and ends with
// exactly one tile segment, so no CTA stops mid-stream to hand on a tile.
//
// Data movement: a producer warp copies the packed weights into a ring of
// shared-memory stages of four consecutive units (32 KB, contiguous in the
// device layout: one bulk asynchronous copy, mbarrier transaction counts),
// as far ahead as the ring allows, so a CTA has most of its bytes requested
// at once and the loads never wait on the arithmetic.  One copy per stage
// rather than per 8 KB unit: measured on gate_up at M = 1, 8.6 against
// 10.5 us.
// Each thread loads its column's fp16 scale and zero word itself, two units
// ahead of use.
//
// Arithmetic: four consumer warpgroups take the CTA's units in turn (unit i
// goes to warpgroup i % 4), thread t column t: four 128-bit shared loads give
// its 128 codes, so one barrier wait, one release and one scale / zero step
// serve 128 weights.  Per token, dot = sum_k (128 + q_k) x_k with the
// bfloat16 value 128 + q made by one mask-and-or per pair of rows (exact) and
// bf16 x bf16 -> f32 fused multiply-adds; then the zero point and scale are
// applied once per group in f32: acc += s (dot - (128 + z) sum_k x_k), with
// the per-group activation sums computed once per CTA.  The scale is used at
// its full binary16 precision.
//
// Reduction: at the end of each tile segment the four warpgroups' sums are
// added through shared memory in warpgroup order.  A tile that lies whole in
// the CTA's range is written directly; a tile shared by several CTAs leaves
// one partial per CTA in the workspace, and the last CTA to arrive on the
// tile's counter adds them in CTA order (deterministic) and writes y.
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
    int split;      // 0: CTA b takes tiles [b NB / P, (b+1) NB / P); 1: tiles are cut into pieces
    int base, extra;  // split: tile t has base + (t < extra) pieces; CTAs are numbered tile by tile
    int S;          // ring stages
    int prefetch;   // weights may be loaded before the preceding grid completes
    int guH;        // > 0: fused gate/up weights (N = 2 guH); y[M][guH] = silu(gate) * up
};

constexpr int kGemvConsumerWarps = 16;                       // four warpgroups
constexpr int kGemvThreads = 32 * (kGemvConsumerWarps + 1);  // plus the producer warp
constexpr int kGemvUnit = 8192;                              // packed weights of one unit, W * 64 bytes
constexpr int kStageUnits = 4;                               // units per stage: one per warpgroup
constexpr int kGemvStage = kStageUnits * kGemvUnit;          // unit j of a stage at j * 8 KB
constexpr int kGemvMaxStages = 8;
constexpr int kGemvMaxSmem = 226 * 1024;

// Pieces of tile t, and the first CTA of tile t (split mode).
__device__ __forceinline__ int tile_pieces(int t, const GemvParams& p) { return p.base + (t < p.extra ? 1 : 0); }
__device__ __forceinline__ int tile_first_cta(int t, const GemvParams& p) {
    return t * p.base + (t < p.extra ? t : p.extra);
}
// The CTA's range of units [ub, ue).
__device__ __forceinline__ void cta_range(int b, const GemvParams& p, int& ub, int& ue) {
    if (!p.split) {
        const int P = (int)gridDim.x;
        ub = (int)((long long)b * p.NB / P) * p.KB;
        ue = (int)((long long)(b + 1) * p.NB / P) * p.KB;
        return;
    }
    const int big = p.extra * (p.base + 1);  // CTAs of the tiles with one piece more
    int t, j, s;
    if (b < big) {
        t = b / (p.base + 1);
        j = b - t * (p.base + 1);
        s = p.base + 1;
    } else {
        t = p.extra + (b - big) / p.base;
        j = (b - big) - (t - p.extra) * p.base;
        s = p.base;
    }
    ub = t * p.KB + (j * p.KB) / s;
    ue = t * p.KB + ((j + 1) * p.KB) / s;
}

__device__ __forceinline__ void consumer_bar() { asm volatile("bar.sync 1, %0;" ::"n"(32 * kGemvConsumerWarps) : "memory"); }

// Shared-memory layout (bytes from the dynamic base), identical on both
// sides.  Every region starts on a 16-byte boundary (the mbarriers need 8).
struct GemvSmem {
    size_t xs, xsum, red, bars, total;
    static __host__ __device__ size_t up16(size_t v) { return (v + 15) & ~(size_t)15; }
    __host__ __device__ GemvSmem(int M, int K, int S) {
        xs = (size_t)S * kGemvStage;                    // ring first (16-byte aligned stages)
        xsum = up16(xs + (size_t)M * K * 2);            // [M][K] bf16 activations
        red = up16(xsum + (size_t)M * (K / 128) * 4);   // [M][K/128] per-group activation sums
        bars = up16(red + (size_t)4 * M * 128 * 4);     // [4][M][128] warpgroup partial sums
        total = bars + (size_t)(2 * S + 1) * 8;         // full[S], empty[S], activations landed
    }
};

template <int M>
__global__ void __launch_bounds__(kGemvThreads, 1) gemv_kernel(const GemvParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int S = p.S;
    const GemvSmem lay(M, p.K, S);
    unsigned char* ring = smem;
    uint16_t* xs = reinterpret_cast<uint16_t*>(smem + lay.xs);
    float* xsum = reinterpret_cast<float*>(smem + lay.xsum);
    float* red = reinterpret_cast<float*>(smem + lay.red);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + lay.bars);
    uint64_t* empty = full + S;
    uint64_t* xbar = empty + S;
    __shared__ int sh_abort, sh_last;
    volatile int* abort_flag = &sh_abort;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const Layout L(p.K, p.N);
    int ub, ue;
    cta_range(blockIdx.x, p, ub, ue);

    if (threadIdx.x < S) {
        mbar_init(&full[threadIdx.x], 1);  // the producer's expect-tx arrival
        fence_mbar_init();
    } else if (threadIdx.x >= 32 && threadIdx.x < 32 + S) {
        mbar_init(&empty[threadIdx.x - 32], 16);  // one arrival per consumer warp
        fence_mbar_init();
    }
    if (threadIdx.x == 64) {
        sh_abort = 0;
        mbar_init(xbar, 1);  // the producer's expect-tx arrival for the activation copy
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kGemvConsumerWarps) {
        // ------------------------------------------------------------ producer
        // The activations (written by the preceding grid) are one bulk copy,
        // the first thing sent once that grid has completed.  With static
        // weights a ring-full of weight copies goes out before that wait
        // (weights, scales and zeros are never written by the preceding grid).
        if (elect_one()) {
            bool x_sent = false;
            auto send_x = [&]() {
                pdl_wait();
                mbar_arrive_expect_tx(xbar, (uint32_t)p.M * p.K * 2);
                bulk_g2s(xs, p.x, (uint32_t)p.M * p.K * 2, xbar);
                x_sent = true;
            };
            if (!p.prefetch) send_x();
            int nb = ub / p.KB, kb = ub - nb * p.KB;
            int s = 0, wraps = 0;  // the next stage is use number `wraps` of stage s
            int issued = 0;
            for (int u = ub; u < ue; u += kStageUnits) {
                if (wraps > 0 && !x_sent) send_x();  // before the first wait on the consumers
                // stage s is free once every consumer warp released its previous use
                if (wraps > 0 && !mbar_wait(&empty[s], (uint32_t)(wraps - 1) & 1u, abort_flag, &g_gemv_status)) {
                    *abort_flag = 1;
                    break;
                }
                const int n = ue - u < kStageUnits ? ue - u : kStageUnits;
                unsigned char* st = ring + (size_t)s * kGemvStage;
                // bytes first (the expected transaction count), then the copies:
                // a run of full-width units is contiguous in memory and lands
                // with one copy; a unit of the ragged last tile has its own
                uint32_t bytes = 0;
                {
                    int tnb = nb, tkb = kb;
                    for (int j = 0; j < n; ++j) {
                        bytes += (uint32_t)L.width(tnb) * 64;
                        if (++tkb == p.KB) { tkb = 0; ++tnb; }
                    }
                }
                mbar_arrive_expect_tx(&full[s], bytes);
                int j = 0;
                while (j < n) {
                    const int W = L.width(nb);
                    const uint32_t* src = p.qd + L.block_word(nb, kb);
                    int run = 1;
                    if (W == 128) {  // following units of full tiles (this tile or the next ones)
                        int tnb = nb, tkb = kb;
                        while (j + run < n) {
                            if (++tkb == p.KB) { tkb = 0; ++tnb; }
                            if (L.width(tnb) != 128) break;
                            ++run;
                        }
                    }
                    bulk_g2s(st + (size_t)j * kGemvUnit, src, (uint32_t)(run * W) * 64, &full[s]);
                    j += run;
                    for (int k = 0; k < run; ++k)
                        if (++kb == p.KB) { kb = 0; ++nb; }
                }
                ++issued;
                if (++s == S) {
                    s = 0;
                    ++wraps;
                }
            }
            if (!x_sent) send_x();
            // every copy issued must land before the CTA may exit
            (void)mbar_wait(xbar, 0, nullptr, &g_gemv_status);
            const int first = issued > S ? issued - S : 0;
            for (int i = first; i < issued; ++i) (void)mbar_wait(&full[i % S], (i / S) & 1, nullptr, &g_gemv_status);
        }
        __syncwarp();
        pdl_launch_dependents();
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int wg = warp >> 2;              // warpgroup 0..3: takes the CTA's units i with i % 4 == wg
    const int t = (warp & 3) * 32 + lane;  // column within the tile
    const int ct = threadIdx.x;            // 0..511
    bool ok = true;
    pdl_wait();  // y and the workspace are written only after the preceding grid
    {
        // rows m >= M of the activations are zero; the others come from the
        // producer's copy; then the per-group sums
        uint4* xv = reinterpret_cast<uint4*>(xs);
        for (int i = p.M * p.K / 8 + ct; i < M * p.K / 8; i += 32 * kGemvConsumerWarps) xv[i] = make_uint4(0, 0, 0, 0);
        if (!mbar_wait_warp(xbar, 0, abort_flag, &g_gemv_status)) ok = false;
        consumer_bar();
        // one group (128 values) per warp: two words per lane, then a butterfly
        for (int i = warp; i < M * p.KB; i += kGemvConsumerWarps) {
            const uint32_t* xr = reinterpret_cast<const uint32_t*>(xs) + (size_t)i * 64;
            const uint32_t v0 = xr[lane], v1 = xr[lane + 32];
            float a = (bf16lo(v0) + bf16hi(v0)) + (bf16lo(v1) + bf16hi(v1));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xFFFFFFFFu, a, o);
            if (lane == 0) xsum[i] = a;
        }
        consumer_bar();
    }
    pdl_launch_dependents();  // one wave: the next grid can only start where this one ends

    // 32-bit shared addresses
    const uint32_t ring_a = smem_u32(smem);
    const uint32_t xs_a = ring_a + (uint32_t)lay.xs;
    const uint32_t xsum_a = ring_a + (uint32_t)lay.xsum;
    const uint32_t full_a = ring_a + (uint32_t)lay.bars;  // full[s] at full_a + 8 s
    const uint32_t empty_a = full_a + 8u * (uint32_t)S;
    const uint32_t xrow = (uint32_t)p.K * 2;             // bytes between token rows of xs
    const uint32_t srow = (uint32_t)p.KB * 4;            // bytes between token rows of xsum
    // independent accumulation chains per 32-row chunk and token: one per
    // word for few tokens, one per chunk when the tokens already give the ILP
    constexpr int NCH = M <= 2 ? 4 : 1;
    int i = wg;  // this warpgroup's next unit, relative to the CTA's first
    int s = 0;   // its stage: unit i is unit i % 4 of stage i / 4 of the walk
    const uint32_t half = (uint32_t)wg * kGemvUnit;
    // scale and zero word of this thread's column for the warpgroup's units,
    // loaded two units ahead of use: (sc0, zw0) for unit i, (sc1, zw1) for i + 4
    int pv = ub + wg;  // next unit to fetch
    int pnb = pv / p.KB, pkb = pv - pnb * p.KB;
    // the column's scale and zero-word pointers at group pkb of tile pnb; four
    // units on they move four groups down, unless the unit is in a later tile
    const uint16_t* sp = nullptr;
    const uint32_t* zp = nullptr;
    auto aim = [&]() {
        const int Wp = L.width(pnb);
        const int tp = t < Wp ? t : Wp - 1;
        const int n = 128 * pnb + tp;
        const int cn = p.guH ? gu_column(n, p.guH) : n;  // canonical column of the scale and zero
        sp = p.scales + (size_t)pkb * p.N + cn;
        zp = p.qzeros + (size_t)pkb * (p.N / 8) + (cn >> 3);
    };
    if (pv < ue) aim();
    const size_t sstep = (size_t)4 * p.N, zstep = (size_t)p.N / 2;
    auto fetch = [&](uint16_t& sc, uint32_t& zw) {
        if (pv < ue) {
            sc = __ldg(sp);
            zw = __ldg(zp);
        }
        pv += 4;
        pkb += 4;
        if (pkb < p.KB) {
            sp += sstep;
            zp += zstep;
        } else {
            do {
                pkb -= p.KB;
                ++pnb;
            } while (pkb >= p.KB);
            if (pv < ue) aim();
        }
    };
    uint16_t sc0 = 0, sc1 = 0;
    uint32_t zw0 = 0, zw1 = 0;
    fetch(sc0, zw0);
    fetch(sc1, zw1);
    uint32_t ph = 0;
    int u = ub;
    int nb = ub / p.KB;
    while (u < ue) {
        // ---- one tile segment: units [u, seg_end) of tile nb
        const int seg_end = ue < (nb + 1) * p.KB ? ue : (nb + 1) * p.KB;
        const int W = L.width(nb);
        const int tc = t < W ? t : W - 1;  // threads beyond a ragged tile read column W-1 and discard it
        const uint32_t w_off = (uint32_t)tc * 16;
        const uint32_t cstep = (uint32_t)W * 16;  // bytes between the unit's 32-row chunks
        const uint32_t zsh = 4u * (uint32_t)(tc & 7);
        const int t0u = nb * p.KB;
        float acc[M];
#pragma unroll
        for (int m = 0; m < M; ++m) acc[m] = 0.f;
        for (; ub + i < seg_end; i += 4) {
            const int kb = ub + i - t0u;
            const uint32_t st_a = ring_a + (uint32_t)s * kGemvStage + half;
            if (ok) {
                const bool ready = mbar_try_wait(full_a + 8u * (uint32_t)s, ph);
                if (!__all_sync(0xFFFFFFFFu, ready) &&
                    !mbar_wait_warp(&full[s], ph, abort_flag, &g_gemv_status))
                    ok = false;
            }
            if (ok) {
                uint4 wc[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) wc[c] = lds_v4(st_a + w_off + (uint32_t)c * cstep);
                const float sc = f16_bits_to_f32(sc0);
                const float zoff = 128.f + (float)((zw0 >> zsh) & 0xFu);
                const uint32_t x_a = xs_a + (uint32_t)kb * 256;
                float d[4 * NCH][M];
#pragma unroll
                for (int c = 0; c < 4 * NCH; ++c)
#pragma unroll
                    for (int m = 0; m < M; ++m) d[c][m] = 0.f;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint32_t wv[4] = {wc[c].x, wc[c].y, wc[c].z, wc[c].w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {  // word j of chunk c: rows 32c + 8j .. +7
                        const int ci = c * NCH + j % NCH;
                        uint32_t wp[4];
#pragma unroll
                        for (int qq = 0; qq < 4; ++qq) wp[qq] = magic_pair(wv[j], qq);
#pragma unroll
                        for (int m = 0; m < M; ++m) {
                            const uint4 xq = lds_v4(x_a + (uint32_t)m * xrow + (uint32_t)(64 * c + 16 * j));
                            const uint32_t xp[4] = {xq.x, xq.y, xq.z, xq.w};
                            float a = d[ci][m];
#pragma unroll
                            for (int qq = 0; qq < 4; ++qq) {
                                a = fma_lo(wp[qq], xp[qq], a);
                                a = fma_hi(wp[qq], xp[qq], a);
                            }
                            d[ci][m] = a;
                        }
                    }
                }
                const uint32_t xz_a = xsum_a + (uint32_t)kb * 4;
#pragma unroll
                for (int m = 0; m < M; ++m) {
                    // pairwise sum of the chains
#pragma unroll
                    for (int w2 = 1; w2 < 4 * NCH; w2 *= 2)
#pragma unroll
                        for (int c = 0; c + w2 < 4 * NCH; c += 2 * w2) d[c][m] += d[c + w2][m];
                    const float xz = __uint_as_float(lds_u32(xz_a + (uint32_t)m * srow));
                    acc[m] = fmaf(sc, fmaf(-zoff, xz, d[0][m]), acc[m]);
                }
            }
            sc0 = sc1;
            zw0 = zw1;
            fetch(sc1, zw1);
            // this warp is done with the stage (its shared loads have returned)
            if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(empty_a + 8u * (uint32_t)s) : "memory");
            if (++s == S) {  // the warpgroup's next unit, four on, is in the next stage
                s = 0;
                ph ^= 1;
            }
        }
        // ---- end of the segment: add the warpgroups, write or hand on
        {
            const int t1u = t0u + p.KB;
            const bool whole = ub <= t0u && ue >= t1u;
            const int n = 128 * nb + t;
#pragma unroll
            for (int m = 0; m < M; ++m) red[(wg * M + m) * 128 + t] = acc[m];
            consumer_bar();
            for (int m = wg; m < M; m += 4) {
                const float v = ((red[(0 * M + m) * 128 + t] + red[(1 * M + m) * 128 + t]) +
                                 red[(2 * M + m) * 128 + t]) + red[(3 * M + m) * 128 + t];
                if (whole) {
                    if (p.guH) {
                        // thread t (t % 16 < 8) holds a gate column, thread t + 8 its up column
                        const float u = __shfl_xor_sync(0xFFFFFFFFu, v, 8);
                        if (!(t & 8) && m < p.M)
                            p.y[(size_t)m * p.guH + gu_column(n, p.guH)] = f32_to_bf16_rn(silu_mul(v, u));
                    } else if (t < W && m < p.M) {
                        p.y[(size_t)m * p.N + n] = f32_to_bf16_rn(v);
                    }
                } else {
                    p.partials[((size_t)blockIdx.x * M + m) * 128 + t] = v;  // one partial per CTA
                }
            }
            if (!whole) {
                // Hand-off: the barrier orders the CTA's partial stores before
                // thread 0, whose gpu-scope fence publishes them with its
                // arrival; the last arrival's fence makes every CTA's
                // partials visible to this CTA after the next barrier.
                consumer_bar();
                const int cf = tile_first_cta(nb, p), cl = cf + tile_pieces(nb, p) - 1;
                if (ct == 0) {
                    __threadfence();
                    const unsigned old = atomicAdd(&p.counters[nb], 1u);
                    const int last = old == (unsigned)(cl - cf);
                    if (last) __threadfence();
                    sh_last = last;
                }
                consumer_bar();
                if (sh_last) {
                    for (int m = wg; m < M; m += 4) {
                        // all partials requested before any is added; then added in CTA order
                        constexpr int kBatch = 8;
                        float sum = 0.f;
                        for (int c0 = cf; c0 <= cl; c0 += kBatch) {
                            float v[kBatch];
#pragma unroll
                            for (int i = 0; i < kBatch; ++i) {
                                const int c = c0 + i;
                                v[i] = 0.f;
                                if (c <= cl) v[i] = __ldcg(p.partials + ((size_t)c * M + m) * 128 + t);
                            }
#pragma unroll
                            for (int i = 0; i < kBatch; ++i)
                                if (c0 + i <= cl) sum += v[i];
                        }
                        if (p.guH) {
                            const float u = __shfl_xor_sync(0xFFFFFFFFu, sum, 8);
                            if (!(t & 8) && m < p.M)
                                p.y[(size_t)m * p.guH + gu_column(n, p.guH)] = f32_to_bf16_rn(silu_mul(sum, u));
                        } else if (t < W && m < p.M) {
                            p.y[(size_t)m * p.N + n] = f32_to_bf16_rn(sum);
                        }
                    }
                    if (ct == 0) p.counters[nb] = 0u;
                }
            }
            consumer_bar();  // red and sh_last are reused by the next segment
        }
        u = seg_end;
        ++nb;
    }
    if (!ok) *abort_flag = 1;
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

static int gemv_mtile(int M) { return M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : 8; }

bool gemv_plan(int M, int N, int K, int sms, GemvPlan* out) {
    if (M < 1 || M > 8 || sms < 1) return false;
    const int MT = gemv_mtile(M);
    const Layout L(K, N);
    const long long U = (long long)L.NB * L.KB;
    if (U < 1 || U >= (1ll << 31)) return false;
    if ((size_t)L.NB > kMaxCounters) return false;
    int ctas, split = 0, base = 0, extra = 0;
    long long per;  // most units of any CTA
    if (L.NB >= sms) {
        ctas = sms;
        per = (long long)((L.NB + sms - 1) / sms) * L.KB;
    } else {
        split = 1;
        if ((long long)L.NB * L.KB <= sms) {  // one unit per CTA
            base = L.KB;
            extra = 0;
            ctas = L.NB * L.KB;
        } else {
            base = sms / L.NB;  // < KB here
            extra = sms % L.NB;
            ctas = sms;
        }
        per = (L.KB + base - 1) / base;
    }
    const size_t fixed = GemvSmem(MT, K, 0).total;
    const size_t per_stage = kGemvStage + 16;
    if (fixed + per_stage > (size_t)kGemvMaxSmem) return false;
    long long S = (long long)(((size_t)kGemvMaxSmem - fixed) / per_stage);
    if (S > kGemvMaxStages) S = kGemvMaxStages;
    long long want = (per + kStageUnits - 1) / kStageUnits;  // stages a CTA uses
    if (want < 2) want = 2;  // one stage filling while another is consumed
    if (S > want) S = want;  // (one stage when no more fits: correct, without overlap)
    const GemvSmem lay(MT, K, (int)S);
    if (lay.xsum % 16 || lay.red % 16 || lay.bars % 16) return false;  // never: regions are rounded up
    out->ctas = ctas;
    out->P = ctas;
    out->C = U;
    out->S = (int)S;
    out->split = split;
    out->base = base;
    out->extra = extra;
    out->smem = lay.total;
    out->ws_bytes = ws_counter_bytes(L.NB) + (size_t)ctas * MT * 128 * sizeof(float);
    return true;
}

template <int M>
static cudaError_t launch_m(const GemvParams& prm, const GemvPlan& plan, cudaStream_t s, bool pdl) {
    auto kern = gemv_kernel<M>;
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
    return launch_kernel(kern, dim3(plan.ctas), dim3(kGemvThreads), plan.smem, s, pdl, prm);
}

cudaError_t launch_gemv(const uint16_t* x, const uint32_t* qd, const uint16_t* scales, const uint32_t* qzeros,
                        uint16_t* y, int M, int N, int K, void* ws, const GemvPlan& plan, cudaStream_t s,
                        unsigned flags, int guH) {
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
    prm.split = plan.split;
    prm.base = plan.base;
    prm.extra = plan.extra;
    prm.S = plan.S;
    const bool pdl = (flags & W4A16_FLAG_PDL) != 0;
    prm.prefetch = pdl && (flags & W4A16_FLAG_STATIC_WEIGHTS) ? 1 : 0;
    prm.guH = guH;
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
