// Tensor-core W4A16 GEMM on sm_103a: persistent, TMA + tcgen05, weights in TMEM.
//
// y[m][n] = sum_g s[g][n] * sum_{k in g} x[m][k] (q[k][n] - z[g][n]), g = 128
// rows: the INT4 linear layer of "Quantize the Target, Quantize the Drafter"
// (pith.science review, referee report summary: AWQ INT4 target with kept
// per-group scales; "Assumptions & free parameters": group size 128), here
// for the 16-token verify blocks (DFlash block size 16) and for prefill.
//
// Orientation (swap AB): the MMA's M = 128 rows are 128 output columns n,
// its N = NT columns are NT tokens.  Work units are (column tile, token tile,
// K split); each CTA walks units blockIdx.x, +gridDim.x, ... and all of its
// roles walk the same sequence of (unit, group) pairs, numbered q = 0, 1, ...
// One pipeline stage carries one group of 128 rows of K.
//
//  * weight producer warp: per group, into weight stage q % SW, the packed
//    weight slab (one bulk copy, 8 KB for a full tile); per chunk of 16
//    groups, the chunk's fp16 scales and zero-point words (2-D tensor
//    copies); activation producer warp: into activation stage q % SX, the x
//    tile (one 3-D TMA, two 64-wide 128-byte swizzled slabs);
//  * dequant warpgroups (four for NT <= 64, two for NT = 128 / 192), taking groups
//    in turn: thread t copies column t's 16 words to registers (releasing
//    the weight stage), turns them into 64 bfloat16 pairs (q - z) -- exact
//    small integers: mask-and-or to 128 + q, subtract 128 + z -- and writes
//    them to tensor memory as the MMA's A operand (tcgen05.st, buffer q % SA);
//    its arrival on the group's "ready" barrier follows the activations'
//    landing too;
//  * two MMA warps, taking groups in turn: each waits for the group's one
//    "ready" barrier (A buffer written, activations landed, D buffer read
//    out), issues its 8 tcgen05.mma kind::f16
//    (A from tensor memory, B = x from shared memory) into D buffer q % NDB
//    and commits them to the group's barrier;
//  * rescale warpgroup(s): per group, reads D with tcgen05.ld and adds
//    s[g][n] * D into f32 registers (the binary16 scale is applied in f32,
//    never rounded to bfloat16); at a unit's end writes bf16 y (with 192-token
//    tiles through shared memory, 16 tokens at a time, as 16-byte rows; for
//    fused gate/up weights silu(gate) * up), or f32 split-K partials, reduced in
//    piece order by the last CTA to arrive -- by the whole CTA once its roles
//    are done when that piece is the CTA's last unit and NT <= 32.
//
// For NT >= 128 a rescale thread holds 64 or 96 accumulators: its warpgroups raise
// their register budget (setmaxnreg) with registers the dequant warpgroups and
// the MMA / producer warpgroup give back, so nothing spills.
//
// Every wait is bounded (common.cuh).  After a timeout every role keeps
// walking its loop without doing work, so all barriers still meet; the CTA
// then drains its copies and MMAs, frees its tensor memory and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"

namespace w4a16 {

static __device__ int g_tc_status;
// Per-thread register budget of the calling warpgroup (all four warps execute
// the same one).  A decrease returns registers to the CTA's pool, an increase
// waits until the pool holds them: the budgets of all warpgroups together must
// not exceed the registers the CTA was launched with.
template <int N>
W4A16_DEVICE void regs_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
W4A16_DEVICE void regs_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

struct TcParams {
    const uint32_t* qd;
    const uint16_t* scales;
    const uint32_t* qzeros;
    uint16_t* y;
    uint32_t* counters;
    float* partials;
    int M, N, K, G;
    int NB, MT;
    int whole;       // units [0, whole) are whole tiles: unit u is tile u
    int splits;      // units from `whole` on: each later tile in `splits` K pieces
    int units;       // whole + (tiles - whole) * splits
    // n / splits and n / NB by multiply and shift (FastDiv below; every role
    // decodes each unit, and four dependent divisions took ~0.4 us)
    uint32_t msplits, mnb;
    int ssplits, snb;
    int prefetch;    // weights may be loaded before the preceding grid completes
    int guH;         // > 0: fused gate/up weights (N = 2 guH); y[M][guH] = silu(gate) * up
    int zmap;        // tmap_z describes the zero words (N % 32 == 0); otherwise the lanes copy them
    int ymap;        // y is 16-byte aligned: whole tiles leave through shared memory in 16-byte rows (NT = 192)
};

// Groups of K per activation stage (the box of the activations' tensor map
// spans 2 XP slabs of 64 columns).
__host__ __device__ constexpr int tc_xp(int) { return 1; }

// Configuration per token-tile width NT.  Weights and activations travel in
// two rings: a weight stage is released by the
// dequant warps as soon as they hold its words in registers, an activation
// stage only when the MMAs reading it are done, so the weight stream runs
// ahead of the tensor core.  A weight stage holds WP consecutive groups of a
// unit (one bulk copy), an activation stage XP.  Both are one: measured on
// the decoder's shapes at M = 16, two groups per stage (one 16 KB copy for
// two weight slabs, one TMA for two activation tiles) made the verify step
// slower (41.4 -> 42.8 us).  The groups' scales and zero words arrive in
// chunks of GB groups (four 2-D tensor copies per chunk, MB chunk buffers),
// issued by the weight producer as it enters a chunk and released by the
// rescale warps after the chunk's last group: measured, per-thread 4-byte
// scale loads kept 16 deep stalled the rescale warps for ~2 us at the start
// and ~0.3 us per group while the weight stream saturated the memory system.
template <int NT>
struct TcCfg {
    static constexpr int R = NT >= 64 ? 2 : 1;           // rescale warpgroups, each owning NT/R columns
    static constexpr int WP = 1;                         // groups per weight stage (1 or 2)
    static constexpr int XP = tc_xp(NT);                 // groups per activation stage
    static constexpr int SX = NT <= 16 ? 12 : NT <= 32 ? 10 : NT <= 64 ? 6 : NT <= 128 ? 4 : 3;  // activation stages
    static constexpr int SW = NT <= 16 ? 16 : NT <= 32 ? 12 : NT <= 64 ? 10 : NT <= 128 ? 8 : 6;  // weight stages
    static constexpr int SA = NT <= 64 ? 4 : NT <= 128 ? 3 : 2;  // A buffers in tensor memory (q % SA)
    static constexpr int NDB = ((512 - SA * 64) / NT) < 8 ? ((512 - SA * 64) / NT) : 8;  // D accumulator ring
    static constexpr int kDone = 16;                     // ring of "MMAs of group q done" barriers
    // ring of "group q may be issued" barriers: its A buffer written and its D
    // buffer read out (arrivals for q follow the completion of q - SA and of
    // q - NDB, so max(SA, NDB) slots keep the phases apart)
    static constexpr int kReady = SA > NDB ? SA : NDB;
    static constexpr int GB = 16;                        // groups per metadata chunk
    static constexpr int MB = 3;                         // metadata chunk buffers
    static constexpr int kDeqWG = NT <= 64 ? 4 : 2;     // dequant warpgroups, taking groups q % kDeqWG
    static constexpr int kDeqWarps = 4 * kDeqWG;
    static constexpr int kResWarp0 = kDeqWarps;          // rescale warpgroups follow
    static constexpr int kMmaIssuers = 2;                // MMA warps, taking groups q % 2
    static constexpr int kMmaWarp = kDeqWarps + 4 * R;   // then the first MMA warp
    static constexpr int kProdWarp = kMmaWarp + 1;       // weight producer (also owns TMEM)
    static constexpr int kXWarp = kProdWarp + 1;         // activation producer
    static constexpr int kMmaWarp2 = kXWarp + 1;         // the second MMA warp
    // NT >= 128: a rescale thread holds 64 or 96 f32 accumulators, more than an even
    // share of the register file allows, so the rescale warpgroups take
    // registers from the other roles (setmaxnreg).  Every role is then whole
    // warpgroups: the last one is the two MMA warps and the two producers.
    static constexpr bool kRegSplit = NT >= 128;
    static constexpr int kWarps = kRegSplit ? (kMmaWarp2 + 4) / 4 * 4 : kMmaWarp2 + 1;
    static constexpr int kThreads = 32 * kWarps;
    static constexpr int kRegDeq = 64, kRegRes = 144, kRegMisc = 64;  // per thread, after the split
    static constexpr int kRegPool =
        32 * (kDeqWarps * kRegDeq + 4 * R * kRegRes + (kWarps - kDeqWarps - 4 * R) * kRegMisc);
    static_assert(!kRegSplit || kRegPool <= kThreads * 96, "register split above a 96-register launch");
    static_assert(!kRegSplit || (kDeqWarps % 4 == 0 && kMmaWarp % 4 == 0), "roles must be whole warpgroups");
    static_assert(SX * XP < kDone && SA <= kDone && NDB <= kDone, "barrier ring too short for the phase parity");
    static_assert(SX * XP >= 2 && SA >= 2 && NDB >= 2, "the two MMA warps' groups need distinct buffers");
    static_assert(2 * SW + SX + 2 * MB + kDone + kReady + 1 <= 128, "barriers are initialised by the first threads");
    static_assert(GB % WP == 0, "a weight stage never straddles two metadata chunks");
    // shared memory, from a 1024-byte aligned base
    static constexpr int kXGroup = NT * 256;             // a group's x: two swizzled boxes of NT rows x 128 bytes
    static constexpr int kXStage = XP * kXGroup;
    static constexpr int kXOff = 0;
    static constexpr int kPOff = kXOff + SX * kXStage;   // packed weights, 8 KB per group
    // metadata chunk: scales [2 boxes][GB groups][64 columns] fp16, then zero
    // words [2 boxes][GB groups][8 words]; box 0 / 1 = the tile's first / second
    // 64 columns (fused gate/up weights: its gate / up columns)
    static constexpr int kMetaScl = 2 * GB * 64 * 2;
    static constexpr int kMetaBytes = kMetaScl + 2 * GB * 8 * 4;
    static constexpr int kMetaOff = kPOff + SW * WP * 8192;
    static constexpr int kBarOff = kMetaOff + MB * kMetaBytes;
    // y staging (NT = 192): per rescale warpgroup two buffers of 16 tokens x
    // 128 columns of bf16, stored as 16-byte rows.  Measured against direct
    // 2-byte stores from the rescale threads: gate_up at M = 2048 174.8 ->
    // 167.0 us (one weight stage fewer to make room); with 16-token tensor
    // stores from the buffers 169.7 us (their reads of shared memory wait
    // behind the activation loads); with 64- and 128-token tiles staging was
    // slightly slower (M = 64, 128), so not used there.
    static constexpr bool kYStore = NT >= 192;
    static constexpr int kYB = 2, kYBytes = 16 * 128 * 2;
    static constexpr int kYOff = kBarOff + 1024;
    static constexpr int kBytes = kYOff + (kYStore ? R * kYB * kYBytes : 0);
    static constexpr int kAlloc = kBytes + 1024;         // slack for the alignment
    // tensor memory: SA A-buffers of 64 columns, then the D ring of NDB x NT columns
    static constexpr int kTmemA = 0;
    static constexpr int kTmemD = SA * 64;
    static constexpr int kTmemUsed = SA * 64 + NDB * NT;
    static constexpr int kTmemCols = kTmemUsed <= 256 ? 256 : 512;
    static_assert(kAlloc <= 227 * 1024, "shared memory budget");
    static_assert(kTmemUsed <= 512, "tensor memory budget");
};

struct UnitInfo {
    int nb, mb, split, ns, g0, g1;
    int ptile;  // for a K piece (ns > 1): index of its tile among the split tiles
};

// Units: the tiles of what would be a partial last round of the persistent
// grid, cut into K pieces spread over all CTAs, come first (so that their
// reductions overlap the rest), then the other tiles whole.  With fewer
// tiles than CTAs every tile is cut (whole = 0).
__device__ __forceinline__ UnitInfo unit_info(const TcParams& p, int u) {
    UnitInfo r;
    int tile;
    const int pieces = p.units - p.whole;
    if (u >= pieces) {
        tile = u - pieces;
        r.split = 0;
        r.ns = 1;
        r.ptile = -1;
    } else {
        r.ptile = div_by(u, p.msplits, p.ssplits);
        r.split = u - r.ptile * p.splits;
        r.ns = p.splits;
        tile = p.whole + r.ptile;
    }
    r.mb = div_by(tile, p.mnb, p.snb);
    r.nb = tile - r.mb * p.NB;
    // (split + 1) G < 2^31 (checked by the planner)
    r.g0 = r.ns == 1 ? 0 : div_by(r.split * p.G, p.msplits, p.ssplits);
    r.g1 = r.ns == 1 ? p.G : div_by((r.split + 1) * p.G, p.msplits, p.ssplits);
    return r;
}

W4A16_DEVICE void tmem_st_x32(uint32_t taddr, const uint32_t* v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
        "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
        "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
        "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}

template <int NT>
__global__ void __launch_bounds__(TcCfg<NT>::kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_s,
                   const __grid_constant__ CUtensorMap tmap_z, const TcParams p) {
    using C = TcCfg<NT>;
    constexpr int SX = C::SX;
    constexpr int SW = C::SW;
    constexpr int SA = C::SA;
    constexpr int R = C::R;
    constexpr int ND = C::kDone;
    // the last unit's split-tile reduction is run by the whole CTA
    constexpr bool kDeferSplit = R == 1 && !C::kRegSplit;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem =
        reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
    uint64_t* wfull = bars;                // [SW] weight stage landed (transactions + cp.async)
    uint64_t* wempty = wfull + SW;         // [SW] weight stage read by its dequant warps
    uint64_t* xfull = wempty + SW;         // [SX] activation stage landed
    uint64_t* mfull = xfull + SX;          // [MB] metadata chunk landed
    uint64_t* mempty = mfull + C::MB;      // [MB] metadata chunk used up by the rescale warps
    uint64_t* done = mempty + C::MB;       // [ND] all MMAs of group q finished: done[q % ND]
    // [kReady] group q may be issued: A buffer q % SA written (4 dequant warps)
    // and D buffer q % NDB read out for group q - NDB (every rescale warp)
    uint64_t* ready = done + ND;
    uint64_t* mma_done = ready + C::kReady;  // [1] every MMA of the CTA finished
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(mma_done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    int* sh_last = const_cast<int*>(abort_flag) + 1;
    // a split tile whose reduction waits for the whole CTA: flag, tile, pieces, first token, column tile
    int* sh_defer = sh_last + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const Layout L(p.K, p.N);

    // barriers initialised in parallel, one per thread
    {
        const int i = threadIdx.x;
        constexpr int MB = C::MB;
        constexpr int nb = 2 * SW + SX + 2 * MB + ND + C::kReady;  // barriers before mma_done
        if (i < SW) mbar_init(&wfull[i], 1);              // the producer's expect-tx arrival
        else if (i < 2 * SW) mbar_init(&wfull[i], 4 * C::WP);  // wempty: four dequant warps per group
        else if (i < 2 * SW + SX) mbar_init(&wfull[i], 1);  // xfull: the producer's expect-tx arrival
        else if (i < 2 * SW + SX + MB) mbar_init(&wfull[i], 1);  // mfull: the producer's expect-tx arrival
        else if (i < 2 * SW + SX + 2 * MB) mbar_init(&wfull[i], 4 * R);  // mempty: every rescale warp
        else if (i < 2 * SW + SX + 2 * MB + ND) mbar_init(&wfull[i], 1);  // done: one MMA commit
        else if (i < nb) mbar_init(&wfull[i], 4 + 4 * R);  // ready
        else if (i == nb) {
            mbar_init(mma_done, C::kMmaIssuers);
            *abort_flag = 0;
            sh_defer[0] = 0;
        }
        if (i <= nb) fence_mbar_init();
    }
    if (warp == C::kProdWarp) {
        tmem_alloc(tmem_holder, C::kTmemCols);
        tmem_relinquish();
        if (lane == 0) {
            prefetch_tmap(&tmap_x);
            prefetch_tmap(&tmap_s);
            if (p.zmap) prefetch_tmap(&tmap_z);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    if (warp != C::kProdWarp && warp != C::kXWarp) pdl_wait();  // producers wait in their own loops

    if (warp >= C::kMmaWarp) {
        // MMA issue, weight and activation producers, and (with the
        // register split) an idle warp: one warpgroup
        if constexpr (C::kRegSplit) regs_dec<C::kRegMisc>();
        if (warp == C::kProdWarp) {
            // ------------------------------------------------ weight producer
            // Per weight stage (WP consecutive groups of a unit): the packed
            // weight slabs in one bulk copy.  On entering a metadata chunk (GB
            // groups of a unit), first the chunk's scales and zero words: 2-D
            // tensor copies of GB rows x 64 columns (two per array), or, for
            // zero words whose rows are not 16-byte aligned (N % 32 != 0),
            // 4-byte asynchronous copies by the lanes.
            constexpr int GB = C::GB, MB = C::MB;
            int wbase = 0, cbase = 0, issued = 0, missued = 0;  // first stage / chunk of the unit; armed
            bool ok = true;
            // This warp touches only weights, scales and zeros: with static
            // weights it never waits on the preceding grid, otherwise once
            // before any load.
            if (!p.prefetch) pdl_wait();
            for (int u = blockIdx.x; u < p.units; u += gridDim.x) {
                const UnitInfo ui = unit_info(p, u);
                const int W = L.width(ui.nb);
                const int Gu = ui.g1 - ui.g0;
                const uint32_t* wsrc = p.qd + L.block_word(ui.nb, ui.g0);
                for (int j = 0; j < Gu; j += C::WP) {
                    if (j % GB == 0) {
                        const int c = cbase + j / GB;
                        const int ms = c % MB;
                        // buffer ms is free once the rescale warps are done with chunk c - MB
                        if (ok && c >= MB &&
                            !mbar_wait_warp(&mempty[ms], ((c - MB) / MB) & 1, abort_flag, &g_tc_status))
                            ok = false;
                        if (ok) {
                            unsigned char* mbuf = smem + C::kMetaOff + ms * C::kMetaBytes;
                            const int g = ui.g0 + j;
                            if (!p.zmap) {
                                // word w of box b, row r: canonical zero word zw(b) + w of group g + r
                                const int zw0 = p.guH ? 8 * ui.nb : 16 * ui.nb;
                                const int zw1 = p.guH ? p.guH / 8 + 8 * ui.nb : 16 * ui.nb + 8;
                                for (int i = lane; i < 2 * GB * 8; i += 32) {
                                    const int b = i / (GB * 8), r = (i / 8) % GB, w = i % 8;
                                    const int zw = (b ? zw1 : zw0) + w;
                                    if (g + r < ui.g1 && zw < p.N / 8)
                                        cp_async_4(mbuf + C::kMetaScl + i * 4, p.qzeros + (size_t)(g + r) * (p.N / 8) + zw);
                                }
                                cp_async_mbar_arrive(&mfull[ms]);
                            }
                            __syncwarp();  // every lane's pending arrival precedes the expected-bytes arrival
                            if (lane == 0) {
                                mbar_arrive_expect_tx(&mfull[ms], (uint32_t)(p.zmap ? C::kMetaBytes : C::kMetaScl));
                                const int sx0 = p.guH ? 64 * ui.nb : 128 * ui.nb;
                                const int sx1 = p.guH ? p.guH + 64 * ui.nb : 128 * ui.nb + 64;
                                tma_load_2d(mbuf, &tmap_s, sx0, g, &mfull[ms]);
                                tma_load_2d(mbuf + GB * 64 * 2, &tmap_s, sx1, g, &mfull[ms]);
                                if (p.zmap) {
                                    const int zx0 = p.guH ? 8 * ui.nb : 16 * ui.nb;
                                    const int zx1 = p.guH ? p.guH / 8 + 8 * ui.nb : 16 * ui.nb + 8;
                                    tma_load_2d(mbuf + C::kMetaScl, &tmap_z, zx0, g, &mfull[ms]);
                                    tma_load_2d(mbuf + C::kMetaScl + GB * 8 * 4, &tmap_z, zx1, g, &mfull[ms]);
                                }
                            }
                            __syncwarp();
                            missued = c + 1;
                        }
                    }
                    const int pw = wbase + j / C::WP;
                    const int s = pw % SW;
                    const int n = Gu - j < C::WP ? Gu - j : C::WP;
                    // stage s is free once the dequant warps of its previous groups hold their words
                    if (ok && pw >= SW &&
                        !mbar_wait_warp(&wempty[s], ((pw - SW) / SW) & 1, abort_flag, &g_tc_status))
                        ok = false;
                    if (ok) {
                        if (lane == 0) {
                            const uint32_t bytes = (uint32_t)(n * W * 64);
                            mbar_arrive_expect_tx(&wfull[s], bytes);
                            bulk_g2s(smem + C::kPOff + s * (C::WP * 8192), wsrc + (size_t)j * W * 16, bytes, &wfull[s]);
                        }
                        __syncwarp();
                        issued = pw + 1;
                    }
                }
                wbase += (Gu + C::WP - 1) / C::WP;
                cbase += (Gu + GB - 1) / GB;
            }
            // drain: every stage and chunk armed must land before the CTA may exit
            for (int i = issued > SW ? issued - SW : 0; i < issued; ++i)
                (void)mbar_wait(&wfull[i % SW], (i / SW) & 1, nullptr, &g_tc_status);
            for (int i = missued > MB ? missued - MB : 0; i < missued; ++i)
                (void)mbar_wait(&mfull[i % MB], (i / MB) & 1, nullptr, &g_tc_status);
        } else if (warp == C::kXWarp) {
            // -------------------------------------------- activation producer
            // Per activation stage (XP consecutive groups of a unit, or fewer at
            // its end): x[tile tokens][128 XP rows of K] with one 3-D TMA
            // (64-wide, 128-byte swizzled slabs; slabs past K read as zeros).
            // Always after the preceding grid.  A stage is refilled once the
            // MMAs of every group it held are done.
            pdl_wait();
            int xbase = 0, issued = 0, q = 0;
            int qwaited = 0;   // groups before this one have had their "done" waited on
            int rend[SX];      // per stage: the flat index one past its last group
            bool ok = true;
            for (int u = blockIdx.x; u < p.units; u += gridDim.x) {
                const UnitInfo ui = unit_info(p, u);
                const int Gu = ui.g1 - ui.g0;
                for (int j = 0; j < Gu; j += C::XP) {
                    const int px = xbase + j / C::XP;
                    const int s = px % SX;
                    const int n = Gu - j < C::XP ? Gu - j : C::XP;
                    if (px >= SX)
                        for (; ok && qwaited < rend[s]; ++qwaited)
                            if (!mbar_wait_warp(&done[qwaited % ND], (qwaited / ND) & 1, abort_flag, &g_tc_status))
                                ok = false;
                    if (ok) {
                        if (lane == 0) {
                            mbar_arrive_expect_tx(&xfull[s], (uint32_t)C::kXStage);
                            tma_load_3d(smem + C::kXOff + s * C::kXStage, &tmap_x, 0, ui.mb * NT, 2 * (ui.g0 + j),
                                        &xfull[s]);
                        }
                        __syncwarp();
                        rend[s] = q + j + n;
                        issued = px + 1;
                    }
                }
                q += Gu;
                xbase += (Gu + C::XP - 1) / C::XP;
            }
            for (int i = issued > SX ? issued - SX : 0; i < issued; ++i)
                (void)mbar_wait(&xfull[i % SX], (i / SX) & 1, nullptr, &g_tc_status);
        } else if (warp == C::kMmaWarp || warp == C::kMmaWarp2) {
            // ------------------------------------------------------------ MMA issue
            // Two MMA warps take the groups in turn, q % 2.  Each runs its loop
            // with all 32 lanes (operands computed by the warp, each instruction
            // issued by one elected lane).  Measured on GB300 at M = 128, N = 16:
            // a warp that waits on a barrier between its groups of 8 MMAs issues
            // one every ~32 ns, whatever the depth it waits at (each wait costs
            // ~190 ns), and two such warps on one SM one every ~16 ns between
            // them; a single lane running the loop alone, one every ~47 ns.
            // Groups q and q + 1 use different A and D buffers and x stages
            // (SA, NDB >= 2), so the two warps' MMAs never touch the same
            // tensor memory; each commit covers the MMAs of its own warp.
            constexpr uint32_t idesc = idesc_bf16_f32(128, NT);
            const int w = warp == C::kMmaWarp ? 0 : 1;
            int q = 0, xbase = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
                const UnitInfo ui = unit_info(p, u);
                const int Gu = ui.g1 - ui.g0;
                for (int j = 0; j < Gu; ++j, ++q) {
                    if ((q % C::kMmaIssuers) != w) continue;
                    // A buffer q % SA written, activations landed, D buffer q % NDB free
                    if (!mbar_wait_warp(&ready[q % C::kReady], (q / C::kReady) & 1, abort_flag, &g_tc_status)) {
                        *abort_flag = 1;
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int px = xbase + j / C::XP;
                    const uint32_t xaddr =
                        smem_u32(smem + C::kXOff + (px % SX) * C::kXStage + (j % C::XP) * C::kXGroup);
                    const uint32_t a_tmem = tmem + C::kTmemA + (q % SA) * 64;
                    const uint32_t d_tmem = tmem + C::kTmemD + (q % C::NDB) * NT;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint64_t bdesc = smem_desc_sw128(xaddr + (kk >> 2) * (NT * 128) + (kk & 3) * 32);
                        mma_bf16_ts_warp(d_tmem, a_tmem + kk * 8, bdesc, idesc, kk > 0 ? 1u : 0u);
                    }
                    mma_commit_warp(&done[q % ND]);
                }
                xbase += (Gu + C::XP - 1) / C::XP;
            }
            // every MMA issued must be complete before TMEM is freed (both
            // warps arrive on mma_done)
            mma_commit_warp(mma_done);
            __syncwarp();
            pdl_launch_dependents();  // this CTA issues no more tensor work
            (void)mbar_wait(mma_done, 0, nullptr, &g_tc_status);
        }
    } else if (warp < C::kDeqWarps) {
        if constexpr (C::kRegSplit) regs_dec<C::kRegDeq>();
        // ------------------------------------------------------------ dequant
        const int h = warp >> 2;              // warpgroup: takes groups q with q % kDeqWG == h
        const int quad = warp & 3;            // TMEM lane quadrant
        const int t = quad * 32 + lane;       // A row = tile column
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        int q = 0, wbase = 0, xbase = 0, cbase = 0;
        int cwaited = -1;  // the last metadata chunk this warp waited for
        bool ok = true;
        for (int u = blockIdx.x; u < p.units; u += gridDim.x) {
            const UnitInfo ui = unit_info(p, u);
            const int W = L.width(ui.nb);
            const int Gu = ui.g1 - ui.g0;
            // columns beyond a ragged tile read column W-1; their A rows only
            // feed D rows that are never written out
            const int tc = t < W ? t : W - 1;
            // this column's zero word in a metadata chunk: box and word index
            const int zbox = p.guH ? (tc >> 3) & 1 : tc >> 6;
            const int zwrd = p.guH ? tc >> 4 : (tc >> 3) & 7;
            for (int j = 0; j < Gu; ++j, ++q) {
                if ((q % C::kDeqWG) != h) continue;
                const int ck = cbase + j / C::GB;  // metadata chunk
                if (ck != cwaited) {
                    if (ok && !mbar_wait_warp(&mfull[ck % C::MB], (ck / C::MB) & 1, abort_flag, &g_tc_status)) ok = false;
                    cwaited = ck;
                }
                const int pw = wbase + j / C::WP, slot = j % C::WP;
                const int s = pw % SW;
                const bool alone = Gu - (j - slot) < C::WP;  // the stage holds this group only
                if (ok && !mbar_wait_warp(&wfull[s], (pw / SW) & 1, abort_flag, &g_tc_status)) ok = false;
                // the column's 128 codes (four 16-byte words) and its zero point
                // into registers, then the group's share of the weight stage goes
                // back to the producer
                uint4 wq[4];
                uint32_t zz = 0x43004300u;
                if (ok) {
                    const uint32_t src = smem_u32(smem + C::kPOff + s * (C::WP * 8192) + slot * W * 64);
#pragma unroll
                    for (int c = 0; c < 4; ++c) wq[c] = lds_v4(src + (uint32_t)((c * W + tc) * 16));
                    const uint32_t zs = smem_u32(smem + C::kMetaOff + (ck % C::MB) * C::kMetaBytes + C::kMetaScl);
                    const uint32_t zw = lds_u32(zs + (uint32_t)(((zbox * C::GB + j % C::GB) * 8 + zwrd) * 4));
                    const uint32_t z = (zw >> (4 * (tc & 7))) & 0xFu;
                    zz = 0x43004300u | z | (z << 16);  // bfloat16 pair (128 + z, 128 + z)
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&wempty[s]);
                        if (alone) mbar_arrive(&wempty[s]);  // the absent group's share
                    }
                }
                uint32_t a[32];
                auto dequant_half = [&](int half) {
#pragma unroll
                    for (int cl = 0; cl < 2; ++cl) {
                        const uint4 v = wq[2 * half + cl];
                        const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                        for (int j = 0; j < 4; ++j)
#pragma unroll
                            for (int pp = 0; pp < 4; ++pp) a[16 * cl + 4 * j + pp] = bf16x2_sub(magic_pair(wv[j], pp), zz);
                    }
                };
                // first half computed before waiting for the A buffer, so the
                // ALU work overlaps the previous group's MMAs
                if (ok) dequant_half(0);
                // A buffer q % SA is free once the MMAs of group q - SA are done
                if (ok && q >= SA &&
                    !mbar_wait_warp(&done[(q - SA) % ND], ((q - SA) / ND) & 1, abort_flag, &g_tc_status))
                    ok = false;
                if (ok) {
                    tc_fence_after();
                    const uint32_t abase = tmem + lane_base + C::kTmemA + (q % SA) * 64;
                    tmem_st_x32(abase, a);
                    tmem_wait_st();  // the registers of the first half are reused below
                    dequant_half(1);
                    tmem_st_x32(abase + 32, a);
                    tmem_wait_st();
                }
                // the group's activations have landed: the MMA warp, which waits
                // only for "ready", reads them after this arrival
                const int px = xbase + j / C::XP;
                if (ok && !mbar_wait_warp(&xfull[px % SX], (px / SX) & 1, abort_flag, &g_tc_status)) ok = false;
                if (ok) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&ready[q % C::kReady]);
                }
                if (!ok) *abort_flag = 1;
            }
            wbase += (Gu + C::WP - 1) / C::WP;
            xbase += (Gu + C::XP - 1) / C::XP;
            cbase += (Gu + C::GB - 1) / C::GB;
        }
    } else {
        if constexpr (C::kRegSplit) regs_inc<C::kRegRes>();
        // ------------------------------------------------------- rescale + epilogue
        const int r = (warp - C::kResWarp0) >> 2;  // rescale warpgroup: owns columns [r*CW, (r+1)*CW)
        const int quad = warp & 3;
        const int t = quad * 32 + lane;
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        constexpr int CW = NT / R;                 // columns (tokens) per rescale warpgroup
        // columns read from tensor memory per wait: all of them where registers allow
        constexpr int kBatch = CW <= 32 || (C::kRegSplit && CW <= 64) ? CW : C::kRegSplit ? 32 : 16;
        const int rt = r * 128 + t;                // thread index among the rescale warpgroups
        float2 acc[CW / 2];
#pragma unroll
        for (int j = 0; j < CW / 2; ++j) acc[j] = make_float2(0.f, 0.f);
        // the D buffers of the first NDB groups start out free
        if (lane == 0)
            for (int i = 0; i < C::NDB; ++i) mbar_arrive(&ready[i]);
        int q = 0, cbase = 0;
        int ych = 0;  // y chunks this warpgroup has staged (buffer ych % kYB)
        bool ok = true;
        // this column's scale in a metadata chunk: box and index
        const int sbox = p.guH ? (t >> 3) & 1 : t >> 6;
        const int sidx = p.guH ? (t >> 4) * 8 + (t & 7) : t & 63;
        for (int u = blockIdx.x; u < p.units; u += gridDim.x) {
            const UnitInfo ui = unit_info(p, u);
            const int W = L.width(ui.nb);
            const int Gu = ui.g1 - ui.g0;
            for (int j = 0; j < Gu; ++j, ++q) {
                const int b = q % C::NDB;
                const int c = cbase + j / C::GB, row = j % C::GB;
                if (row == 0 && ok && !mbar_wait_warp(&mfull[c % C::MB], (c / C::MB) & 1, abort_flag, &g_tc_status))
                    ok = false;
                const uint32_t sa = smem_u32(smem + C::kMetaOff + (c % C::MB) * C::kMetaBytes);
                const float sc = f16_bits_to_f32(lds_u16(sa + (uint32_t)(((sbox * C::GB + row) * 64 + sidx) * 2)));
                if (ok && !mbar_wait_warp(&done[q % ND], (q / ND) & 1, abort_flag, &g_tc_status)) ok = false;
                if (ok) {
                    tc_fence_after();
                    const float2 sc2 = make_float2(sc, sc);
                    const uint32_t dbase = tmem + lane_base + C::kTmemD + b * NT + r * CW;
                    if constexpr (C::kRegSplit && kBatch == CW) {
                        // all columns in one load: the D buffer goes back to the
                        // MMA before the multiply-adds
                        uint32_t v[CW];
#pragma unroll
                        for (int c = 0; c < CW; c += 16)
                            tmem_ld_x16(dbase + c, *reinterpret_cast<uint32_t(*)[16]>(v + c));
                        tmem_wait_ld();
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&ready[(q + C::NDB) % C::kReady]);  // D buffer b free for group q + NDB
#pragma unroll
                        for (int i = 0; i < CW; i += 2)
                            acc[i / 2] = __ffma2_rn(sc2, make_float2(__uint_as_float(v[i]), __uint_as_float(v[i + 1])),
                                                    acc[i / 2]);
                    } else {
#pragma unroll
                        for (int c0 = 0; c0 < CW; c0 += kBatch) {
                            uint32_t v[kBatch];
#pragma unroll
                            for (int c = 0; c < kBatch; c += 16)
                                tmem_ld_x16(dbase + c0 + c, *reinterpret_cast<uint32_t(*)[16]>(v + c));
                            tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < kBatch; i += 2)
                                acc[(c0 + i) / 2] = __ffma2_rn(
                                    sc2, make_float2(__uint_as_float(v[i]), __uint_as_float(v[i + 1])), acc[(c0 + i) / 2]);
                        }
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&ready[(q + C::NDB) % C::kReady]);  // D buffer b free for group q + NDB
                    }
                }
                // the chunk's last group: its buffer goes back to the producer
                if (row == C::GB - 1 || j == Gu - 1) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&mempty[c % C::MB]);
                }
                if (!ok) *abort_flag = 1;
            }
            cbase += (Gu + C::GB - 1) / C::GB;
            // ---- end of unit: this warpgroup writes its CW tokens of the tile
            const bool all_ok = bar_and(4, 128 * R, ok && !*abort_flag);
            const int n = 128 * ui.nb + t;
            const int tok0 = ui.mb * NT + r * CW;
            if (all_ok) {
                if (ui.ns == 1) {
                    if (C::kYStore && p.ymap) {
                        // Per 16 tokens: every thread writes its values into a
                        // staging buffer; after the warpgroup's barrier each thread
                        // stores 16 contiguous bytes of a token row.  Chunk k uses
                        // buffer k % 2: its writes follow the barrier of chunk k - 1,
                        // after which nobody reads chunk k - 2's buffer.  Fused
                        // gate/up weights: a row holds the tile's 64 outputs, thread
                        // t (gate lane, t % 16 < 8) the even tokens of output
                        // 8 (t / 16) + t % 8 and its up lane t + 8 the odd ones.
                        unsigned char* ybase = smem + C::kYOff + r * (C::kYB * C::kYBytes);
#pragma unroll
                        for (int c = 0; c < CW / 16; ++c) {
                            if (tok0 + 16 * c >= p.M) break;  // uniform in the warpgroup
                            const uint32_t buf = smem_u32(ybase + (ych & 1) * C::kYBytes);
                            if (p.guH) {
                                const bool gate = !(t & 8);
                                const int oc = 8 * (t >> 4) + (t & 7);
#pragma unroll
                                for (int i = 0; i < 16; i += 2) {
                                    const float a0 = acc[(16 * c + i) / 2].x, a1 = acc[(16 * c + i) / 2].y;
                                    const float o = __shfl_xor_sync(0xFFFFFFFFu, gate ? a1 : a0, 8);
                                    const int row = i + (gate ? 0 : 1);
                                    sts_u16(buf + (uint32_t)(row * 128 + 2 * oc),
                                            f32_to_bf16_rn(gate ? silu_mul(a0, o) : silu_mul(o, a1)));
                                }
                                named_bar(6 + r, 128);
                                const int row = t >> 3, tok = tok0 + 16 * c + row;
                                const uint4 v = lds_v4(buf + (uint32_t)(row * 128 + 16 * (t & 7)));
                                if (tok < p.M)
                                    *reinterpret_cast<uint4*>(p.y + (size_t)tok * p.guH + 64 * ui.nb + 8 * (t & 7)) = v;
                            } else {
                                const int cx = 8 * (t & 15);  // this thread's columns in the row
#pragma unroll
                                for (int i = 0; i < 16; ++i) {
                                    const int j = 16 * c + i;
                                    sts_u16(buf + (uint32_t)(i * 256 + 2 * t),
                                            f32_to_bf16_rn((j & 1) ? acc[j / 2].y : acc[j / 2].x));
                                }
                                named_bar(6 + r, 128);
#pragma unroll
                                for (int h = 0; h < 2; ++h) {
                                    const int row = (t >> 4) + 8 * h;
                                    const int tok = tok0 + 16 * c + row;
                                    const int col = 128 * ui.nb + cx;
                                    const uint4 v = lds_v4(buf + (uint32_t)(row * 256 + 2 * cx));
                                    if (tok < p.M && col < p.N)  // N % 8 == 0: all 8 columns or none
                                        *reinterpret_cast<uint4*>(p.y + (size_t)tok * p.N + col) = v;
                                }
                            }
                            ++ych;
                        }
                    } else if (p.guH) {
                        // Thread t (t % 16 < 8) holds a gate column, thread t + 8 its
                        // up column.  Per pair of tokens one value crosses each way: the
                        // gate lane finishes token j, the up lane token j + 1.
                        const bool gate = !(t & 8);
                        const size_t col = (size_t)gu_column(gate ? n : n - 8, p.guH);
#pragma unroll
                        for (int j = 0; j < CW; j += 2) {
                            const float a0 = acc[j / 2].x, a1 = acc[j / 2].y;  // tokens j, j + 1
                            const float r = __shfl_xor_sync(0xFFFFFFFFu, gate ? a1 : a0, 8);
                            const int tok = tok0 + j + (gate ? 0 : 1);
                            if (tok < p.M)
                                p.y[(size_t)tok * p.guH + col] = f32_to_bf16_rn(gate ? silu_mul(a0, r) : silu_mul(r, a1));
                        }
                    } else if (t < W) {
#pragma unroll
                        for (int j = 0; j < CW; ++j)
                            if (tok0 + j < p.M)
                                p.y[(size_t)(tok0 + j) * p.N + n] =
                                    f32_to_bf16_rn((j & 1) ? acc[j / 2].y : acc[j / 2].x);
                    }
                } else {
                    const int tile = ui.ptile;  // counters and partials of the split tiles only
                    // partial sums: [split tile][piece][NT / 4][128 columns][4 tokens]: a
                    // thread writes (and the reduction reads) four tokens of its column
                    // as one 16-byte vector, a warp 512 contiguous bytes
                    float4* part = reinterpret_cast<float4*>(p.partials) +
                                   (((size_t)tile * ui.ns + ui.split) * (NT / 4) + r * (CW / 4)) * 128 + t;
#pragma unroll
                    for (int j = 0; j < CW / 4; ++j)
                        part[(size_t)j * 128] =
                            make_float4(acc[2 * j].x, acc[2 * j].y, acc[2 * j + 1].x, acc[2 * j + 1].y);
                    // hand-off: the barrier orders the warpgroups' partial stores
                    // before one thread, whose gpu-scope fence publishes them
                    // with its arrival; the last arrival fences again before
                    // the barrier that releases the reduction
                    asm volatile("bar.sync 5, %0;" ::"r"(128 * R) : "memory");
                    if (rt == 0) {
                        __threadfence();
                        const unsigned old = atomicAdd(&p.counters[tile], 1u);
                        const int last = old == (unsigned)ui.ns - 1;
                        if (last) __threadfence();
                        *sh_last = last;
                    }
                    asm volatile("bar.sync 5, %0;" ::"r"(128 * R) : "memory");
                    // Only with one rescale warpgroup (NT <= 32), where its own
                    // reduction needs the most round trips per element; never with
                    // the register split, where every warp would run it, also those
                    // that gave registers away.
                    const bool last_unit = kDeferSplit && u + (int)gridDim.x >= p.units;
                    if (*sh_last && last_unit) {
                        // the CTA's last unit: every warp of the CTA joins the
                        // reduction once the roles are done (more loads in flight)
                        if (rt == 0) {
                            sh_defer[1] = tile;
                            sh_defer[2] = ui.ns;
                            sh_defer[3] = ui.mb * NT;
                            sh_defer[4] = ui.nb;
                            sh_defer[0] = 1;
                        }
                    } else if (*sh_last) {
                        // every split's values for this thread, summed in split order,
                        // TJ tokens at a time with the loads of two pieces in flight
                        // together.  The reduction is latency-bound: 16 tokens a pass
                        // held the reducing CTA ~9.6 us on a three-piece 192-token
                        // tile; 32 a pass (where the register split leaves room) took
                        // the prefill step 348 -> 345 us, three pieces a round spilled
                        // and was slower (359 us).
                        constexpr int TJ = C::kRegSplit ? 32 : 16;
                        constexpr int PK = 2;
                        const float4* base = reinterpret_cast<const float4*>(p.partials) +
                                             ((size_t)tile * ui.ns * (NT / 4) + r * (CW / 4)) * 128 + t;
                        const size_t sstride = (size_t)(NT / 4) * 128;  // float4s between splits
#pragma unroll 1
                        for (int j0 = 0; j0 < CW; j0 += TJ) {
                            float4 sum[TJ / 4];
#pragma unroll
                            for (int i = 0; i < TJ / 4; ++i) sum[i] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
                            for (int sp0 = 0; sp0 < ui.ns; sp0 += PK) {
                                float4 v[PK][TJ / 4];
#pragma unroll
                                for (int k = 0; k < PK; ++k)
#pragma unroll
                                    for (int i = 0; i < TJ / 4; ++i)
                                        v[k][i] = sp0 + k < ui.ns
                                                      ? __ldcg(base + (sp0 + k) * sstride + (size_t)(j0 / 4 + i) * 128)
                                                      : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                                for (int k = 0; k < PK; ++k)
                                    if (sp0 + k < ui.ns)
#pragma unroll
                                        for (int i = 0; i < TJ / 4; ++i) {
                                            sum[i].x += v[k][i].x;
                                            sum[i].y += v[k][i].y;
                                            sum[i].z += v[k][i].z;
                                            sum[i].w += v[k][i].w;
                                        }
                            }
                            if (p.guH) {
                                const bool gate = !(t & 8);
                                const size_t col = (size_t)gu_column(gate ? n : n - 8, p.guH);
#pragma unroll
                                for (int j = 0; j < TJ; j += 2) {
                                    const float4& v = sum[j / 4];
                                    const float a0 = (j & 2) ? v.z : v.x, a1 = (j & 2) ? v.w : v.y;
                                    const float r = __shfl_xor_sync(0xFFFFFFFFu, gate ? a1 : a0, 8);
                                    const int jj = j0 + j + (gate ? 0 : 1);
                                    if (jj < CW && tok0 + jj < p.M)
                                        p.y[(size_t)(tok0 + jj) * p.guH + col] =
                                            f32_to_bf16_rn(gate ? silu_mul(a0, r) : silu_mul(r, a1));
                                }
                            } else if (t < W) {
#pragma unroll
                                for (int j = 0; j < TJ; ++j) {
                                    const float4& v = sum[j / 4];
                                    const float val = (j & 3) == 0 ? v.x : (j & 3) == 1 ? v.y : (j & 3) == 2 ? v.z : v.w;
                                    if (j0 + j < CW && tok0 + j0 + j < p.M)
                                        p.y[(size_t)(tok0 + j0 + j) * p.N + n] = f32_to_bf16_rn(val);
                                }
                            }
                        }
                        if (rt == 0) p.counters[tile] = 0u;
                    }
                    asm volatile("bar.sync 5, %0;" ::"r"(128 * R) : "memory");  // sh_last is reused
                }
            }
#pragma unroll
            for (int j = 0; j < CW / 2; ++j) acc[j] = make_float2(0.f, 0.f);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == C::kProdWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
    if constexpr (kDeferSplit) {
    if (sh_defer[0] && !*abort_flag) {
        // Deferred reduction of a split tile by every thread of the CTA: element
        // e of a piece's partials ([NT / 4][128 columns][4 tokens]) is summed
        // over the pieces in piece order, the loads of up to kE elements and
        // kS pieces in flight at once.  kS = 4 rather than 8 (smaller code, run
        // once per launch): verify step 37.35 -> 37.03 us; kE = 2: 38.54 us.
        constexpr int kE = 3, kS = 4;
        const int tile = sh_defer[1], ns = sh_defer[2], tokb = sh_defer[3], nbt = sh_defer[4];
        const int W = L.width(nbt);
        const float* base = p.partials + (size_t)tile * ns * NT * 128;
        const int nthr = (int)blockDim.x;
        const int nel = p.guH ? NT * 64 : NT * 128;  // gate/up: one element per gate column
        for (int e0 = (int)threadIdx.x; e0 < nel; e0 += kE * nthr) {
            int ea[kE];
            float sum[kE], sup[kE];
#pragma unroll
            for (int k = 0; k < kE; ++k) {
                const int i = e0 + k * nthr;
                if (p.guH) {  // i -> (token quad, gate column with bit 3 clear, token)
                    const int jj = i % 4, rc = i / 4, tq = rc / 64, c64 = rc % 64;
                    ea[k] = i < nel ? (tq * 128 + (c64 / 8) * 16 + (c64 % 8)) * 4 + jj : -1;
                } else {
                    ea[k] = i < nel ? i : -1;
                }
                sum[k] = 0.f;
                sup[k] = 0.f;
            }
            for (int sp0 = 0; sp0 < ns; sp0 += kS) {
                float v[kE][kS], vu[kE][kS];
#pragma unroll
                for (int k = 0; k < kE; ++k)
#pragma unroll
                    for (int q2 = 0; q2 < kS; ++q2) {
                        const bool in = ea[k] >= 0 && sp0 + q2 < ns;
                        const float* pp = base + (size_t)(sp0 + q2) * NT * 128 + ea[k];
                        v[k][q2] = in ? __ldcg(pp) : 0.f;
                        vu[k][q2] = in && p.guH ? __ldcg(pp + 8 * 4) : 0.f;
                    }
#pragma unroll
                for (int k = 0; k < kE; ++k)
#pragma unroll
                    for (int q2 = 0; q2 < kS; ++q2)
                        if (sp0 + q2 < ns) {
                            sum[k] += v[k][q2];
                            sup[k] += vu[k][q2];
                        }
            }
#pragma unroll
            for (int k = 0; k < kE; ++k) {
                if (ea[k] < 0) continue;
                const int col = (ea[k] / 4) % 128;
                const int tok = tokb + (ea[k] / 512) * 4 + ea[k] % 4;
                if (tok >= p.M) continue;
                const int n = 128 * nbt + col;
                if (p.guH)
                    p.y[(size_t)tok * p.guH + gu_column(n, p.guH)] = f32_to_bf16_rn(silu_mul(sum[k], sup[k]));
                else if (col < W)
                    p.y[(size_t)tok * p.N + n] = f32_to_bf16_rn(sum[k]);
            }
        }
        if (threadIdx.x == 0) p.counters[tile] = 0u;
    }
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
// Token tile when neither the caller nor the dispatch table names one (the
// table's measured choices follow the same steps): the smallest tile that
// holds M up to 64 tokens, 128 up to 256, then 192 -- two D buffers of 192
// columns still fit beside two A buffers in the 512 tensor-memory columns, and
// the larger tile reads each weight slab for more tokens.
static int tc_nt(int M) { return M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : M <= 256 ? 128 : 192; }

bool tc_plan(int M, int N, int K, int sms, TcPlan* out, int force_nt) {
    const Layout L(K, N);
    const int G = K / 128;
    if (force_nt && force_nt != 16 && force_nt != 32 && force_nt != 64 && force_nt != 128 && force_nt != 192)
        return false;
    const int table_nt = force_nt ? 0 : dispatch_nt(M, K, N);
    const int NT = force_nt ? force_nt : table_nt ? table_nt : tc_nt(M);
    const int MT = (M + NT - 1) / NT;
    const long long slots = sms;  // CTAs resident at once, one per SM
    const long long tiles = (long long)L.NB * MT;
    const int max_split = G / 2 > 0 ? G / 2 : 1;  // at least 2 groups a piece
    long long whole = tiles;
    // Pieces of a partial last round for K of at least 16 groups, at least 5
    // groups each.  Measured at M = 2048 with the earlier token-major partials: the
    // 4096-deep tiles of o_proj 50.1 -> 45.9 us (two pieces), the 2560-deep
    // tiles of qkv unchanged (three pieces), the 9728-deep ones of down as
    // with pieces of 8 or more.
    const int max_split_tail = G >= 16 ? G / 5 : 1;
    int splits = 1;
    if (tiles < slots) {
        // Fewer tiles than CTAs: every tile in K pieces, rounded down so that
        // no CTA runs two units while others idle.
        const long long s = slots / tiles < max_split ? slots / tiles : max_split;
        if (s > 1) {
            splits = (int)s;
            whole = 0;
        }
    } else if (tiles % slots) {
        // Full rounds of whole tiles; the tiles of the partial last round in
        // K pieces spread over all CTAs.
        const long long rem = tiles % slots;
        const long long s = slots / rem < max_split_tail ? slots / rem : max_split_tail;
        if (s > 1) {
            splits = (int)s;
            whole = tiles - rem;
        }
    }
    if (tiles - whole > (long long)kMaxCounters) {  // counters for the split tiles
        whole = tiles;
        splits = 1;
    }
    const long long units = whole + (tiles - whole) * splits;
    if (units >= (1ll << 31) || tiles >= (1ll << 31) || (long long)splits * G >= (1ll << 31)) return false;
    out->NT = NT;
    out->MT = MT;
    out->NB = L.NB;
    out->whole = (int)whole;
    out->splits = splits;
    out->units = (int)units;
    out->ctas = (int)(units < slots ? units : slots);
    out->smem = NT == 16    ? TcCfg<16>::kAlloc
                : NT == 32  ? TcCfg<32>::kAlloc
                : NT == 64  ? TcCfg<64>::kAlloc
                : NT == 128 ? TcCfg<128>::kAlloc
                            : TcCfg<192>::kAlloc;
    const long long split_tiles = tiles - whole;
    out->ws_bytes = split_tiles > 0
                        ? ws_counter_bytes((size_t)split_tiles) + (size_t)split_tiles * splits * NT * 128 * sizeof(float)
                        : 0;
    return true;
}

static PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

template <int NT>
static cudaError_t launch_nt(const CUtensorMap& tm, const CUtensorMap& tms, const CUtensorMap& tmz, const TcParams& prm,
                             const TcPlan& plan, cudaStream_t s, bool pdl) {
    using C = TcCfg<NT>;
    auto kern = tc_gemm_kernel<NT>;
    static int set_for[64];  // shared memory limit raised once per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!set_for[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kAlloc);
        if (e != cudaSuccess) return e;
        if (C::kRegSplit) {
            // the warpgroups' register budgets must fit in what the CTA is
            // launched with, or the increase would wait forever: never launch then
            cudaFuncAttributes fa;
            e = cudaFuncGetAttributes(&fa, kern);
            if (e != cudaSuccess) return e;
            if ((long long)fa.numRegs * C::kThreads < C::kRegPool) return cudaErrorInvalidConfiguration;
        }
        set_for[dev] = 1;
    }
    return launch_kernel(kern, dim3(plan.ctas), dim3(C::kThreads), plan.smem, s, pdl, tm, tms, tmz, prm);
}


cudaError_t launch_tc(const uint16_t* x, const uint32_t* qd, const uint16_t* scales, const uint32_t* qzeros,
                      uint16_t* y, int M, int N, int K, void* ws, const TcPlan& plan, cudaStream_t s,
                      unsigned flags, int guH) {
    auto encode = get_encode();
    if (!encode) return cudaErrorNotSupported;
    CUtensorMap tm;
    // x viewed as [K/64 slabs][M tokens][64 columns]: one box is NT tokens x
    // 2 XP slabs of 64 columns, i.e. XP groups of 128 rows of K
    const cuuint64_t dims[3] = {64, (cuuint64_t)M, (cuuint64_t)(K / 64)};
    const cuuint64_t strides[2] = {(cuuint64_t)K * 2, 128};
    const cuuint32_t box[3] = {64, (cuuint32_t)plan.NT, (cuuint32_t)(2 * tc_xp(plan.NT))};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = encode(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(x), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    // scales [G][N] fp16 and zero words [G][N/8]: boxes of 16 groups (the
    // metadata chunk) x 64 columns / 8 words
    constexpr int GB = TcCfg<16>::GB;
    static_assert(TcCfg<16>::GB == TcCfg<192>::GB, "one chunk height for every token tile");
    CUtensorMap tms, tmz;
    {
        const cuuint64_t sd[2] = {(cuuint64_t)N, (cuuint64_t)(K / 128)};
        const cuuint64_t ss[1] = {(cuuint64_t)N * 2};
        const cuuint32_t sb[2] = {64, GB};
        const cuuint32_t se[2] = {1, 1};
        r = encode(&tms, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<uint16_t*>(scales), sd, ss, sb, se,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    // zero-word rows are N/2 bytes apart: a tensor map needs that to be a multiple of 16
    const int zmap = N % 32 == 0;
    tmz = tms;
    if (zmap) {
        const cuuint64_t zd[2] = {(cuuint64_t)(N / 8), (cuuint64_t)(K / 128)};
        const cuuint64_t zs[1] = {(cuuint64_t)N / 2};
        const cuuint32_t zb[2] = {8, GB};
        const cuuint32_t ze[2] = {1, 1};
        r = encode(&tmz, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint32_t*>(qzeros), zd, zs, zb, ze,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    // staged epilogue of whole tiles (NT = 192): 16-byte rows of y
    const int ymap = plan.NT >= 192 && ((uintptr_t)y & 15) == 0;
    TcParams prm;
    prm.qd = qd;
    prm.scales = scales;
    prm.qzeros = qzeros;
    prm.y = y;
    const size_t split_tiles = (size_t)plan.NB * plan.MT - (size_t)plan.whole;
    prm.counters = reinterpret_cast<uint32_t*>(ws);
    prm.partials = ws ? reinterpret_cast<float*>(reinterpret_cast<char*>(ws) + ws_counter_bytes(split_tiles)) : nullptr;
    prm.M = M;
    prm.N = N;
    prm.K = K;
    prm.G = K / 128;
    prm.NB = plan.NB;
    prm.MT = plan.MT;
    prm.whole = plan.whole;
    prm.splits = plan.splits;
    prm.units = plan.units;
    const FastDiv fs = fast_div(plan.splits), fn = fast_div(plan.NB);
    prm.msplits = fs.m;
    prm.ssplits = fs.s;
    prm.mnb = fn.m;
    prm.snb = fn.s;
    const bool pdl = (flags & W4A16_FLAG_PDL) != 0;
    prm.prefetch = pdl && (flags & W4A16_FLAG_STATIC_WEIGHTS) ? 1 : 0;
    prm.guH = guH;
    prm.zmap = zmap;
    prm.ymap = ymap;
    switch (plan.NT) {
        case 16: return launch_nt<16>(tm, tms, tmz, prm, plan, s, pdl);
        case 32: return launch_nt<32>(tm, tms, tmz, prm, plan, s, pdl);
        case 64: return launch_nt<64>(tm, tms, tmz, prm, plan, s, pdl);
        case 192: return launch_nt<192>(tm, tms, tmz, prm, plan, s, pdl);
        default: return launch_nt<128>(tm, tms, tmz, prm, plan, s, pdl);
    }
}

int tc_read_status() {
    int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_tc_status, sizeof(int)) != cudaSuccess) return W4A16_ECUDA;
    if (cudaMemcpyToSymbol(g_tc_status, &zero, sizeof(int)) != cudaSuccess) return W4A16_ECUDA;
    return v;
}

}  // namespace w4a16
