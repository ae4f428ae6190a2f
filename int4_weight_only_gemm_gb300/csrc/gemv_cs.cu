// Column-sliced GEMV for M = 1..8 on CUDA cores (sm_103a).
//
// y[m][n] = sum_k x[m][k] (q[k][n] - z[g][n]) s[g][n], g = k / 128: the INT4
// linear layer run at every decode step by the quantized target and drafter
// of "Quantize the Target, Quantize the Drafter" (pith.science review,
// referee report summary; group size 128 from "Assumptions & free
// parameters").
//
// Work split: CTA b owns a contiguous slice of columns [c0, c1) over all of K
// (slices are whole units of 4 columns, or 16 for fused gate/up weights so
// that a gate column and its up column stay together), so no CTA ever hands
// a partial sum to another and no workspace is needed.  Inside the CTA,
// thread t takes column j = t % C of the slice and the range s = t / C of
// whole 128-row groups of K (S = min(512 / C, K / 128) ranges), or, for
// slices wider than half the block, whole columns j = t, t + 512, ...
//
// Data movement: the unit of work is an item, one column's 32 rows of K: 16
// bytes of the device layout (word j of chunk c holds rows 8(4c + j)..+7).
// A column's items lie a constant W * 16 bytes apart (W = width of its
// 128-column tile), and the lanes of a warp read adjacent columns, so each
// copy instruction of a warp fetches contiguous runs.  Each thread streams
// its items with 16-byte asynchronous copies into a private ring of D + 1
// shared-memory slots of IPS consecutive items (one commit group a slot), D
// slots ahead of the one it multiplies: the distance is fixed by the copies
// in flight, not by register scheduling, and the wait and ring bookkeeping
// are paid once a slot.  After the grid-dependency wait x goes first, then
// the scales and the first D slots; the multiplication starts once x and the
// first slot are in.
//
// Arithmetic: per item and token, the dot product of the 32 rows with x,
// sum (128 + q) x, with the bfloat16 value 128 + q made by one mask-and-or
// per pair of rows (exact) and bf16 x bf16 -> f32 fused multiply-adds in
// four independent chains; the zero point and scale apply once per 128-row
// group in f32: acc += s (dot - (128 + z) xs), xs = the group's sum of x
// (computed once per CTA).  The scale is used at its full binary16 precision.
// The K ranges of a column are added through shared memory in range order:
// the result does not depend on timing.
//
// Footprint: one CTA per SM with up to 128 registers a thread.  (Capped at 64
// registers, two CTAs fit on an SM and the next programmatic-dependent GEMM
// of a chain becomes resident while this one runs; measured on the decode
// step, that chain is slower: 27.3 against 24.9 us.)
#include "common.cuh"
#include "kernels.h"

namespace w4a16 {

struct CsParams {
    const uint16_t* x;
    const uint32_t* qd;
    const uint16_t* scales;
    const uint32_t* qzeros;
    uint16_t* y;
    int M, N, K, KB;  // KB = K / 128 groups
    int U, unit;      // column units and their width (4, or 16 for fused gate/up)
    int prefetch;     // weights, scales and zeros may be read before the preceding grid completes
    int guH;          // > 0: fused gate/up weights (N = 2 guH); y[M][guH] = silu(gate) * up
    // CTA b owns column units [b U / P, (b + 1) U / P): slices of Cw[0] or
    // Cw[1] columns, with Sr[k] K ranges; the divisions by P, by the slice
    // width, by the range count and by a quarter of the width are multiplies
    // and shifts (FastDiv: four dependent divisions sat between a CTA's start
    // and its first weight copy)
    uint32_t mP;
    int sP;
    int Cw[2], Sr[2];
    uint32_t mC[2], mS[2], mC4[2];
    int sC[2], sS[2], sC4[2];
};

constexpr int kCsThreads = 512;

// Shared-memory layout (bytes from the dynamic base), identical on both
// sides; every region starts on a 16-byte boundary.
struct CsSmem {
    size_t xs, xsum, sc, zr, ring, red, total;
    static __host__ __device__ size_t up16(size_t v) { return (v + 15) & ~(size_t)15; }
    // MT: token rows held (M rounded up), C: slice width, D: ring slots in
    // flight a thread, IPS: items a slot.  Every region grows with C, so the
    // widest slice of a launch sizes it for all its CTAs.
    __host__ __device__ CsSmem(int MT, int K, int C, int D, int IPS) {
        const int G = K / 128;
        xs = 0;                                          // [MT][K] bf16 activations
        xsum = up16(xs + (size_t)MT * K * 2);            // [MT][G] f32 group sums of x
        sc = up16(xsum + (size_t)MT * G * 4);            // [G][C] fp16 scales of the slice
        zr = up16(sc + (size_t)G * C * 2);               // [G][C/4] zero words, one per run of 4 columns
        ring = up16(zr + (size_t)G * C);                       // [D + 1][IPS][512] 16-byte items
        red = ring + (size_t)(D + 1) * IPS * kCsThreads * 16;  // [S][C][MT] f32 partial sums (S C <= max(512, C))
        total = up16(red + (size_t)(C > kCsThreads ? C : kCsThreads) * MT * 4);
    }
};

__host__ __device__ inline int cs_ranges(int C, int G) {
    int S = C >= kCsThreads / 2 ? 1 : kCsThreads / C;
    return S < G ? S : G;
}

template <int MT, int D, int IPS>
__global__ void __launch_bounds__(kCsThreads, 1) gemv_cs_kernel(const CsParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int t = threadIdx.x;
    const int b = blockIdx.x;
    // slice bounds ((b + 1) U < 2^31 and S G < 2^31: checked by the planner)
    const int c0 = p.unit * div_by(b * p.U, p.mP, p.sP);
    const int c1 = p.unit * div_by((b + 1) * p.U, p.mP, p.sP);
    const int C = c1 - c0;
    const int kw = C == p.Cw[0] ? 0 : 1;  // which of the two slice widths
    const int G = p.KB;
    const int S = p.Sr[kw];
    const CsSmem lay(MT, p.K, C, D, IPS);
    uint16_t* xs = reinterpret_cast<uint16_t*>(smem + lay.xs);
    float* xsum = reinterpret_cast<float*>(smem + lay.xsum);
    uint16_t* ssc = reinterpret_cast<uint16_t*>(smem + lay.sc);
    uint32_t* szw = reinterpret_cast<uint32_t*>(smem + lay.zr);
    uint4* ring = reinterpret_cast<uint4*>(smem + lay.ring) + t;  // item i of slot k at ring[(k IPS + i) 512]
    float* red = reinterpret_cast<float*>(smem + lay.red);

    // the next grid in the stream may start as soon as every CTA of this one runs
    pdl_launch_dependents();

    // this thread's work: column j0 (then j0 + 512, ... when S == 1), groups [g0, g1)
    const bool active = t < S * C || S == 1;
    const int s = S == 1 ? 0 : div_by(t, p.mC[kw], p.sC[kw]);
    const int j0 = S == 1 ? t : t - s * C;
    const int g0 = div_by(s * G, p.mS[kw], p.sS[kw]);
    const int g1 = div_by((s + 1) * G, p.mS[kw], p.sS[kw]);
    const int nr = 4 * (g1 - g0);  // items of one column
    const int npass = S == 1 ? (j0 < C ? (C - j0 + kCsThreads - 1) / kCsThreads : 0) : (active ? 1 : 0);
    const int nslots = npass * nr / IPS;  // slot fills (IPS divides 4: a fill never crosses a column)
    const uint4* qd4 = reinterpret_cast<const uint4*>(p.qd);

    // Copy cursor over this thread's items, pass by pass: item r of column n
    // is uint4 512 KB nb + W r + (n % 128) of the device layout (W = width of
    // tile nb), so a column's items are W uint4 apart.
    const uint4* lptr = nullptr;
    int lstride = 0, lp = 0, lr = 0, issued = 0, lslot = 0;
    auto set_column = [&](int pass) {
        const int n = c0 + j0 + pass * kCsThreads;
        const int nb = n >> 7;
        lstride = p.N - 128 * nb < 128 ? p.N - 128 * nb : 128;
        lptr = qd4 + (size_t)512 * p.KB * nb + (size_t)lstride * (4 * g0) + (n & 127);
    };
    // fill `issued` (IPS consecutive items of a column) into its slot, one
    // commit group per fill (possibly empty)
    const bool passes = npass > 1;  // a thread with one column needs no column switch
    auto copy_next = [&]() {
        if (issued < nslots) {
            uint4* dst = ring + (size_t)lslot * (IPS * kCsThreads);
#pragma unroll
            for (int i = 0; i < IPS; ++i) cp_async_16(dst + i * kCsThreads, lptr + i * lstride);
            lslot = lslot == D ? 0 : lslot + 1;
            lptr += IPS * lstride;
            if (passes && (lr += IPS) == nr) {
                lr = 0;
                if (++lp < npass) set_column(lp);
            }
            ++issued;
        }
        cp_async_commit();
    };
    // The slice's scales ([G][C] fp16, device-column order) and, per run of
    // four columns, the zero word holding their zero points ([G][C/4]).  Four
    // adjacent device columns are four adjacent canonical columns in both
    // layouts, and a column's zero nibble sits at bit 4 (n % 8) of its word.
    auto stage_scales_zeros = [&]() {
        const int C4 = C >> 2;
        for (int i = t; i < G * C4; i += kCsThreads) {
            const int g = div_by(i, p.mC4[kw], p.sC4[kw]), jj = 4 * (i - g * C4);
            const int n = c0 + jj;
            const int cn = p.guH ? gu_column(n, p.guH) : n;
            cp_async_8(ssc + (size_t)g * C + jj, p.scales + (size_t)g * p.N + cn);
            cp_async_4(szw + i, p.qzeros + (size_t)g * (p.N / 8) + (cn >> 3));
        }
        cp_async_commit();
    };
    auto start_items = [&]() {
        if (nslots > 0) set_column(0);
#pragma unroll 1
        for (int i = 0; i < D; ++i) copy_next();
    };

    // activations: rows m < M copied (asynchronously), rows M..MT-1 zero
    auto copy_x = [&]() {
        const int n16 = MT * p.K / 8;
        const int v16 = p.M * p.K / 8;
        const uint4* xg = reinterpret_cast<const uint4*>(p.x);
        uint4* xv = reinterpret_cast<uint4*>(xs);
        for (int i = t; i < n16; i += kCsThreads) {
            if (i < v16) cp_async_16(xv + i, xg + i);
            else xv[i] = make_uint4(0, 0, 0, 0);
        }
        cp_async_commit();
    };
    // Commit groups complete in order.  With static weights the first D items
    // and the scales go out before the grid dependency resolves and x after
    // it, so x's group is the newest and all must have landed; otherwise x
    // and the scales go first, and the multiplication starts once they and
    // the first item are in, while the other D - 1 items are still coming.
    if (p.prefetch) {
        start_items();
        stage_scales_zeros();
        pdl_wait();  // x, and y below, only after the preceding grid
        copy_x();
        cp_async_wait<0>();
    } else {
        pdl_wait();
        copy_x();
        stage_scales_zeros();
        start_items();
        cp_async_wait<D>();  // x and the scales (the D slot groups may be pending)
    }
    __syncthreads();
    // per-group activation sums, one (token, group) per warp
    {
        const int warp = t >> 5, lane = t & 31;
        for (int i = warp; i < MT * G; i += kCsThreads / 32) {
            const uint32_t* xr = reinterpret_cast<const uint32_t*>(xs) + (size_t)i * 64;
            const uint32_t v0 = xr[lane], v1 = xr[lane + 32];
            float a = (bf16lo(v0) + bf16hi(v0)) + (bf16lo(v1) + bf16hi(v1));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xFFFFFFFFu, a, o);
            if (lane == 0) xsum[i] = a;
        }
    }
    __syncthreads();

    const uint32_t xs_a = smem_u32(xs);
    const uint32_t ring_a = smem_u32(ring);
    const uint32_t xrow = (uint32_t)p.K * 2;  // bytes between token rows of xs
    constexpr int NCH = MT == 1 ? 4 : 2;  // independent chains a token
    int kslot = 0;                        // ring slot of the items being multiplied
    uint4 wk[IPS];                        // that slot's items
#pragma unroll 1
    for (int pass = 0; pass < npass; ++pass) {
        const int jj = j0 + pass * kCsThreads;
        const uint32_t zsh = 4u * (uint32_t)((c0 + jj) & 7);  // this column's nibble in its zero word
        float acc[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[m] = 0.f;
#pragma unroll 1
        for (int g = g0; g < g1; ++g) {
            float d[MT][NCH];
#pragma unroll
            for (int m = 0; m < MT; ++m)
#pragma unroll
                for (int c = 0; c < NCH; ++c) d[m][c] = 0.f;
#pragma unroll
            for (int it = 0; it < 4; ++it) {  // the group's four items
                if (it % IPS == 0) {
                    cp_async_wait<D - 1>();  // this slot has landed (D - 1 newer fills may be pending)
#pragma unroll
                    for (int i = 0; i < IPS; ++i)
                        wk[i] = lds_v4(ring_a + (uint32_t)(kslot * IPS + i) * (kCsThreads * 16));
                    kslot = kslot == D ? 0 : kslot + 1;
                    copy_next();  // the fill D further on, into the slot the previous one used
                }
                const uint4 w = wk[it % IPS];
                const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
                const int r = 4 * g + it;
#pragma unroll
                for (int q = 0; q < 4; ++q) {  // word q: rows 8q .. 8q + 7 of the item
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        const uint4 xq = lds_v4(xs_a + (uint32_t)m * xrow + (uint32_t)r * 64 + (uint32_t)q * 16);
                        const uint32_t xp[4] = {xq.x, xq.y, xq.z, xq.w};
                        float a = d[m][q % NCH];
#pragma unroll
                        for (int pp = 0; pp < 4; ++pp) {
                            const uint32_t wp = magic_pair(wv[q], pp);
                            a = fma_lo(wp, xp[pp], a);
                            a = fma_hi(wp, xp[pp], a);
                        }
                        d[m][q % NCH] = a;
                    }
                }
            }
            const float sc = f16_bits_to_f32(ssc[g * C + jj]);
            const float zoff = 128.f + (float)((szw[g * (C >> 2) + (jj >> 2)] >> zsh) & 0xFu);
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                // pairwise sum of the chains
#pragma unroll
                for (int w2 = 1; w2 < NCH; w2 *= 2)
#pragma unroll
                    for (int c = 0; c + w2 < NCH; c += 2 * w2) d[m][c] += d[m][c + w2];
                const float dot = d[m][0];
                acc[m] = fmaf(sc, fmaf(-zoff, xsum[m * G + g], dot), acc[m]);
            }
        }
        // this column's sums over this thread's K range
#pragma unroll
        for (int m = 0; m < MT; ++m) red[((size_t)s * C + jj) * MT + m] = acc[m];
    }
    cp_async_wait<0>();  // the trailing commit groups are empty; nothing stays in flight
    __syncthreads();

    // the K ranges of each column added in range order; fused weights: the
    // gate column (device column d, d % 16 < 8) meets its up column d + 8
    for (int i = t; i < C * MT; i += kCsThreads) {
        const int jj = i / MT, m = i - jj * MT;
        if (m >= p.M) continue;
        const int n = c0 + jj;
        if (p.guH) {
            if (n & 8) continue;  // up columns are read by their gate column
            float g = 0.f, u = 0.f;
            for (int r = 0; r < S; ++r) {
                g += red[((size_t)r * C + jj) * MT + m];
                u += red[((size_t)r * C + jj + 8) * MT + m];
            }
            p.y[(size_t)m * p.guH + gu_column(n, p.guH)] = f32_to_bf16_rn(silu_mul(g, u));
        } else {
            float v = 0.f;
            for (int r = 0; r < S; ++r) v += red[((size_t)r * C + jj) * MT + m];
            p.y[(size_t)m * p.N + n] = f32_to_bf16_rn(v);
        }
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

static int cs_mtile(int M) { return M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : 8; }
constexpr int kCsMaxSmem = 226 * 1024;

// Ring of a thread, for up to two tokens: eight items in flight, in fills of
// two items.  Measured on the decode step (M = 1): items one at a time took
// 4.21 / 4.63 / 8.39 / 6.87 us (qkv / o_proj / gate_up / down), fills of two
// 3.87 / 4.37 / 8.20 / 6.67, fills of four 3.86 / 4.12 / 8.52 / 6.67 (fewer
// instructions: 5.00 against 5.92 M on gate_up, but there the coarser waits
// cost more than they save); with the prologue's divisions replaced, fills
// of two everywhere (3.61 / 4.11 / 7.90 / 6.41, step 21.1 us) beat fills of
// four for qkv and o_proj (3.86 / 4.11, step 21.2 us).  More tokens need the
// registers for the products: single items, eight in flight, or four where
// eight would not fit the shared memory.
bool gemv_cs_plan(int M, int N, int K, int sms, int guH, GemvCsPlan* out) {
    if (M < 1 || M > 8 || sms < 1 || K < 128 || K % 128 || N % 8) return false;
    const int unit = guH ? 16 : 4;
    if (N % unit) return false;
    const long long U = N / unit;
    const int P = (int)(U < sms ? U : sms);
    // the kernel's slice arithmetic stays below 2^31: (b + 1) U and S G (S <= 512)
    if ((long long)(P + 1) * U >= (1ll << 31) || (long long)(K / 128) * kCsThreads >= (1ll << 31)) return false;
    const int MT = cs_mtile(M);
    // the widest slice decides the shared memory
    const int C = (int)(unit * ((U + P - 1) / P));
    // (slots in flight, items a slot), in order of preference
    const int forms[3][2] = {{4, 2}, {8, 1}, {4, 1}};
    int f = MT > 2 ? 1 : 0;
    while (f < 3 && CsSmem(MT, K, C, forms[f][0], forms[f][1]).total > (size_t)kCsMaxSmem) ++f;
    if (f == 3) return false;
    const int D = forms[f][0], IPS = forms[f][1];
    const CsSmem lay(MT, K, C, D, IPS);
    out->ctas = P;
    out->U = (int)U;
    out->unit = unit;
    out->D = D;
    out->ips = IPS;
    out->smem = lay.total;
    return true;
}

template <int MT, int D, int IPS>
static cudaError_t launch_cs(const CsParams& prm, const GemvCsPlan& plan, cudaStream_t s, bool pdl) {
    auto kern = gemv_cs_kernel<MT, D, IPS>;
    static int set_for[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!set_for[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kCsMaxSmem);
        if (e != cudaSuccess) return e;
        set_for[dev] = 1;
    }
    return launch_kernel(kern, dim3(plan.ctas), dim3(kCsThreads), plan.smem, s, pdl, prm);
}

template <int MT>
static cudaError_t launch_cs_mt(const CsParams& prm, const GemvCsPlan& plan, cudaStream_t s, bool pdl) {
    if constexpr (MT <= 2) {
        if (plan.ips == 2) return launch_cs<MT, 4, 2>(prm, plan, s, pdl);
    }
    return plan.D == 8 ? launch_cs<MT, 8, 1>(prm, plan, s, pdl) : launch_cs<MT, 4, 1>(prm, plan, s, pdl);
}

cudaError_t launch_gemv_cs(const uint16_t* x, const uint32_t* qd, const uint16_t* scales, const uint32_t* qzeros,
                           uint16_t* y, int M, int N, int K, const GemvCsPlan& plan, cudaStream_t s, unsigned flags,
                           int guH) {
    CsParams prm;
    prm.x = x;
    prm.qd = qd;
    prm.scales = scales;
    prm.qzeros = qzeros;
    prm.y = y;
    prm.M = M;
    prm.N = N;
    prm.K = K;
    prm.KB = K / 128;
    prm.U = plan.U;
    prm.unit = plan.unit;
    const FastDiv fp = fast_div(plan.ctas);
    prm.mP = fp.m;
    prm.sP = fp.s;
    for (int k = 0; k < 2; ++k) {
        const int cw = plan.unit * (plan.U / plan.ctas + k);
        const int sr = cs_ranges(cw, K / 128);
        const FastDiv fc = fast_div(cw), fs = fast_div(sr), fc4 = fast_div(cw / 4);
        prm.Cw[k] = cw;
        prm.Sr[k] = sr;
        prm.mC[k] = fc.m;
        prm.sC[k] = fc.s;
        prm.mS[k] = fs.m;
        prm.sS[k] = fs.s;
        prm.mC4[k] = fc4.m;
        prm.sC4[k] = fc4.s;
    }
    const bool pdl = (flags & W4A16_FLAG_PDL) != 0;
    prm.prefetch = pdl && (flags & W4A16_FLAG_STATIC_WEIGHTS) ? 1 : 0;
    prm.guH = guH;
    switch (cs_mtile(M)) {
        case 1: return launch_cs_mt<1>(prm, plan, s, pdl);
        case 2: return launch_cs_mt<2>(prm, plan, s, pdl);
        case 4: return launch_cs_mt<4>(prm, plan, s, pdl);
        default: return launch_cs_mt<8>(prm, plan, s, pdl);
    }
}

}  // namespace w4a16
