// Tensor-core W4A16 GEMM on sm_103a: TMA + tcgen05 with the weights in TMEM.
//
// y[m][n] = sum_g s[g][n] * sum_{k in g} x[m][k] (q[k][n] - z[g][n]), g = 128
// rows: the INT4 linear layer of "Quantize the Target, Quantize the Drafter"
// (pith.science review, referee report summary: AWQ INT4 target with kept
// per-group scales; "Assumptions & free parameters": group size 128), here
// for the 16-token verify blocks (DFlash block size 16) and for prefill.
//
// Orientation (swap AB): the MMA's M = 128 rows are 128 output columns n,
// its N = NT columns are NT tokens.  D[n][token] lives in tensor memory.
//
//  * producer warp: per 64-row K stage, one bulk copy of the packed weight
//    slab (4 KB, contiguous in the device layout) and one TMA tile of x
//    (NT tokens x 64 bf16, 128-byte swizzle) into a 4-deep shared ring;
//  * dequant warpgroup: thread t turns its column's 8 words into 32 bfloat16
//    pairs (q - z), exact small integers (mask-and-or to 128 + q, subtract
//    128 + z), and writes them to tensor memory as the MMA's A operand
//    (tcgen05.st), so the dequantized weights never touch shared memory;
//  * MMA warp: one thread issues tcgen05.mma kind::f16 (A from TMEM, B = x
//    from shared memory), 4 per stage; each group of 128 rows accumulates
//    into its own D buffer (two, double-buffered);
//  * rescale warpgroup: per group, reads D_g with tcgen05.ld and adds
//    s[g][n] * D_g into f32 registers -- the binary16 scale is applied in
//    f32, never rounded to bfloat16 -- then writes bf16 y (or split-K partials).
//
// Every wait is bounded (see common.cuh); on a timeout the CTA stops, waits
// for its own copies in flight, frees its tensor memory and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"

namespace w4a16 {

static __device__ int g_tc_status;

constexpr int kStages = 4;         // K stages of 64 rows in the ring
constexpr int kStageK = 64;
constexpr int kPackedStageBytes = 128 * kStageK / 2;  // 4 KB
constexpr int kThreads = 320;      // 10 warps: producer, MMA, 4 dequant, 4 rescale

struct TcParams {
    const uint32_t* qd;
    const uint16_t* scales;
    const uint32_t* qzeros;
    uint16_t* y;
    uint32_t* counters;
    float* partials;
    int M, N, K, G;
    int NB, MT;      // column tiles, token tiles
    int splits;      // K splits (groups divided evenly)
    int prefetch;    // weights may be loaded before the preceding grid completes
};

template <int NT>
struct TcSmem {
    static constexpr int kXStage = NT * 128;  // NT rows x 64 bf16
    static constexpr int kXOff = 0;
    static constexpr int kPOff = kXOff + kStages * kXStage;
    static constexpr int kBarOff = kPOff + kStages * kPackedStageBytes;
    static constexpr int kBytes = kBarOff + 256;
    static constexpr int kAlloc = kBytes + 1024;  // slack for 1024-byte alignment
    // tensor memory columns: D double buffer + A ring (32 columns per stage)
    static constexpr int kTmemD = 0;
    static constexpr int kTmemA = 2 * NT;
    static constexpr int kTmemCols = (2 * NT + kStages * 32) <= 256 ? 256 : 512;
};

template <int NT>
__global__ void __launch_bounds__(kThreads, NT <= 32 ? 2 : 1) tc_gemm_kernel(const __grid_constant__ CUtensorMap tmap_x,
                                                              const TcParams p) {
    using S = TcSmem<NT>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem =
        reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kBarOff);
    uint64_t* full = bars;                   // [kStages] tx: packed + x arrived
    uint64_t* a_full = bars + kStages;       // [kStages] A stage written to TMEM
    uint64_t* empty = bars + 2 * kStages;    // [kStages] MMA done with the stage
    uint64_t* d_full = bars + 3 * kStages;   // [2] group accumulated
    uint64_t* d_empty = d_full + 2;          // [2] group read by rescale warps
    uint64_t* mma_done = d_empty + 2;        // [1] every issued MMA has finished
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(mma_done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    int* sh_last = const_cast<int*>(abort_flag) + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nb = blockIdx.x, mb = blockIdx.y, split = blockIdx.z;
    const Layout L(p.K, p.N);
    const int W = L.width(nb);
    const int g_begin = (int)((long long)split * p.G / p.splits);
    const int g_end = (int)((long long)(split + 1) * p.G / p.splits);
    const int n_groups = g_end - g_begin;
    const int n_stages = 2 * n_groups;
    const int tok0 = mb * NT;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&a_full[i], 4);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&d_full[i], 1);
            mbar_init(&d_empty[i], 4);
        }
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, S::kTmemCols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) prefetch_tmap(&tmap_x);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    // everything but the producer thread reads global memory only after the
    // preceding grid has completed (the producer waits in its own loop)
    if (!(warp == 0 && lane == 0)) pdl_wait();

    if (warp == 0) {
        // ---------------- producer ----------------
        if (lane == 0) {
            int issued = 0;
            const uint32_t pbytes = (uint32_t)W * 32;  // W columns x 8 words
            // with static weights, the first ring's weight slabs go out before
            // waiting on the preceding grid; x only after it
            const int pre = p.prefetch ? (n_stages < kStages ? n_stages : kStages) : 0;
            for (int it = 0; it < pre; ++it) {
                const int kb = g_begin + (it >> 1);
                mbar_arrive_expect_tx(&full[it], pbytes + S::kXStage);
                bulk_g2s(smem + S::kPOff + it * kPackedStageBytes,
                         p.qd + L.block_word(nb, kb) + (size_t)(it & 1) * 2 * W * 4, pbytes, &full[it]);
            }
            pdl_wait();
            for (int it = 0; it < n_stages; ++it) {
                const int s = it % kStages;
                const int use = it / kStages;
                const int kb = g_begin + (it >> 1);
                const int half = it & 1;
                if (it >= pre) {
                    if (use > 0 && !mbar_wait(&empty[s], (use - 1) & 1, abort_flag, &g_tc_status)) break;
                    mbar_arrive_expect_tx(&full[s], pbytes + S::kXStage);
                    const uint32_t* src = p.qd + L.block_word(nb, kb) + (size_t)half * 2 * W * 4;
                    bulk_g2s(smem + S::kPOff + s * kPackedStageBytes, src, pbytes, &full[s]);
                }
                tma_load_2d(smem + S::kXOff + s * S::kXStage, &tmap_x, kb * 128 + half * 64, tok0, &full[s]);
                ++issued;
            }
            if (issued < pre) issued = pre;  // prefetched slabs are in flight too
            // drain: every issued stage must have landed before the CTA may exit
            for (int it = (issued > kStages ? issued - kStages : 0); it < issued; ++it) {
                const int s = it % kStages;
                const int use = it / kStages;
                uint64_t t0 = globaltimer();
                while (!mbar_try_wait(smem_u32(&full[s]), use & 1)) {
                    if (globaltimer() - t0 > kWaitNs) {
                        atomicExch(&g_tc_status, (int)W4A16_ETIMEOUT);
                        break;
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(128, NT);
            bool ok = true;
            for (int gi = 0; gi < n_groups && ok; ++gi) {
                const int b = gi & 1;
                const int buse = gi >> 1;
                if (buse > 0 && !mbar_wait(&d_empty[b], (buse - 1) & 1, abort_flag, &g_tc_status)) break;
                tc_fence_after();
                for (int h = 0; h < 2; ++h) {
                    const int it = 2 * gi + h;
                    const int s = it % kStages;
                    const int use = it / kStages;
                    if (!mbar_wait(&full[s], use & 1, abort_flag, &g_tc_status) ||
                        !mbar_wait(&a_full[s], use & 1, abort_flag, &g_tc_status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t xaddr = smem_u32(smem + S::kXOff + s * S::kXStage);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t bdesc = smem_desc_sw128(xaddr + kk * 32);
                        const uint32_t a_tmem = tmem + S::kTmemA + s * 32 + kk * 8;
                        const uint32_t d_tmem = tmem + S::kTmemD + b * NT;
                        mma_bf16_ts(d_tmem, a_tmem, bdesc, idesc, (h | kk) ? 1u : 0u);
                    }
                    mma_commit(&empty[s]);
                }
                if (ok) mma_commit(&d_full[b]);
            }
            pdl_launch_dependents();  // this CTA issues no more work; let the next grid queue up
            // all MMAs this thread issued must be complete before TMEM is freed
            mma_commit(mma_done);
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(smem_u32(mma_done), 0)) {
                if (globaltimer() - t0 > kWaitNs) {
                    atomicExch(&g_tc_status, (int)W4A16_ETIMEOUT);
                    break;
                }
            }
        }
    } else if (warp < 6) {
        // ---------------- dequant warpgroup (warps 2..5) ----------------
        const int quad = warp & 3;          // TMEM lane quadrant this warp may access
        const int t = quad * 32 + lane;     // row of A = column of the tile
        const int n = nb * 128 + t;
        const bool valid = t < W;
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        uint32_t zz = 0x43004300u;
        for (int it = 0; it < n_stages; ++it) {
            const int s = it % kStages;
            const int use = it / kStages;
            const int kb = g_begin + (it >> 1);
            if ((it & 1) == 0 && valid) {
                const uint32_t zw = __ldg(p.qzeros + (size_t)kb * (p.N / 8) + (n >> 3));
                const uint32_t z = (zw >> (4 * (n & 7))) & 0xFu;
                zz = 0x43004300u | z | (z << 16);  // bfloat16 pair (128 + z, 128 + z)
            }
            if (!mbar_wait_warp(&full[s], use & 1, abort_flag, &g_tc_status)) break;
            uint32_t a[32];
            if (valid) {
                const uint4* src = reinterpret_cast<const uint4*>(smem + S::kPOff + s * kPackedStageBytes);
#pragma unroll
                for (int cl = 0; cl < 2; ++cl) {
                    const uint4 v = src[cl * W + t];
                    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j)
#pragma unroll
                        for (int q = 0; q < 4; ++q) a[16 * cl + 4 * j + q] = bf16x2_sub(magic_pair(wv[j], q), zz);
                }
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) a[i] = 0u;
            }
            const uint32_t abase = tmem + lane_base + S::kTmemA + s * 32;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint32_t v8[8] = {a[8 * c], a[8 * c + 1], a[8 * c + 2], a[8 * c + 3],
                                        a[8 * c + 4], a[8 * c + 5], a[8 * c + 6], a[8 * c + 7]};
                tmem_st_x8(abase + 8 * c, v8);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&a_full[s]);
        }
    } else {
        // ---------------- rescale / epilogue warpgroup (warps 6..9) ----------------
        const int quad = warp & 3;
        const int t = quad * 32 + lane;
        const int n = nb * 128 + t;
        const bool valid = t < W;
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        float acc[NT];
#pragma unroll
        for (int j = 0; j < NT; ++j) acc[j] = 0.f;
        float sc = valid ? f16_bits_to_f32(__ldg(p.scales + (size_t)g_begin * p.N + n)) : 0.f;
        bool ok = true;
        for (int gi = 0; gi < n_groups; ++gi) {
            const int b = gi & 1;
            const int buse = gi >> 1;
            const float sc_next =
                (valid && gi + 1 < n_groups) ? f16_bits_to_f32(__ldg(p.scales + (size_t)(g_begin + gi + 1) * p.N + n))
                                             : 0.f;
            if (!mbar_wait_warp(&d_full[b], buse & 1, abort_flag, &g_tc_status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t dbase = tmem + lane_base + S::kTmemD + b * NT;
#pragma unroll
            for (int c = 0; c < NT / 16; ++c) {
                uint32_t v[16];
                tmem_ld_x16(dbase + 16 * c, v);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i) acc[16 * c + i] = fmaf(sc, __uint_as_float(v[i]), acc[16 * c + i]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&d_empty[b]);
            sc = sc_next;
        }
        // every rescale thread reaches this barrier, failed or not, and they
        // agree on whether to write anything
        if (bar_and(1, 128, ok)) {
            const int tile = nb * p.MT + mb;
            if (p.splits == 1) {
                if (valid) {
#pragma unroll
                    for (int j = 0; j < NT; ++j)
                        if (tok0 + j < p.M) p.y[(size_t)(tok0 + j) * p.N + n] = f32_to_bf16_rn(acc[j]);
                }
            } else {
                float* part = p.partials + ((size_t)tile * p.splits + split) * NT * 128;
#pragma unroll
                for (int j = 0; j < NT; ++j) part[j * 128 + t] = acc[j];
                __threadfence();
                asm volatile("bar.sync 2, 128;" ::: "memory");
                if (t == 0) {
                    const unsigned old = atomicAdd(&p.counters[tile], 1u);
                    *sh_last = (old == (unsigned)p.splits - 1) ? 1 : 0;
                }
                asm volatile("bar.sync 2, 128;" ::: "memory");
                if (*sh_last) {
                    __threadfence();
                    const float* base = p.partials + (size_t)tile * p.splits * NT * 128;
#pragma unroll 4
                    for (int j = 0; j < NT; ++j) {
                        float sum = 0.f;
                        for (int sp = 0; sp < p.splits; ++sp) sum += __ldcg(base + ((size_t)sp * NT + j) * 128 + t);
                        if (valid && tok0 + j < p.M) p.y[(size_t)(tok0 + j) * p.N + n] = f32_to_bf16_rn(sum);
                    }
                    if (t == 0) p.counters[tile] = 0u;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, S::kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------


static int tc_nt(int M) { return M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : 128; }

bool tc_plan(int M, int N, int K, int sms, TcPlan* out) {
    const Layout L(K, N);
    const int G = K / 128;
    const int NT = tc_nt(M);
    const int MT = (M + NT - 1) / NT;
    const long long tiles = (long long)L.NB * MT;
    // split K so that the grid covers the SMs about once (at least 2 groups a split)
    int splits = 1;
    if (tiles < sms) {
        splits = (int)((sms + tiles - 1) / tiles);
        const int max_split = G / 2 > 0 ? G / 2 : 1;
        if (splits > max_split) splits = max_split;
    }
    if (splits > 1 && (size_t)tiles > kMaxCounters) splits = 1;
    out->NT = NT;
    out->MT = MT;
    out->NB = L.NB;
    out->splits = splits;
    switch (NT) {
        case 16: out->smem = TcSmem<16>::kAlloc; break;
        case 32: out->smem = TcSmem<32>::kAlloc; break;
        case 64: out->smem = TcSmem<64>::kAlloc; break;
        default: out->smem = TcSmem<128>::kAlloc; break;
    }
    out->ws_bytes = splits > 1 ? ws_counter_bytes(tiles) + (size_t)tiles * splits * NT * 128 * sizeof(float) : 0;
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
static cudaError_t launch_nt(const CUtensorMap& tm, const TcParams& prm, const TcPlan& plan, cudaStream_t s,
                             bool pdl) {
    auto kern = tc_gemm_kernel<NT>;
    static int set_for[64];  // shared memory limit raised once per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!set_for[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)TcSmem<NT>::kAlloc);
        if (e != cudaSuccess) return e;
        set_for[dev] = 1;
    }
    dim3 grid(plan.NB, plan.MT, plan.splits);
    return launch_kernel(kern, grid, dim3(kThreads), plan.smem, s, pdl, tm, prm);
}

cudaError_t launch_tc(const uint16_t* x, const uint32_t* qd, const uint16_t* scales, const uint32_t* qzeros,
                      uint16_t* y, int M, int N, int K, void* ws, const TcPlan& plan, cudaStream_t s,
                      unsigned flags) {
    auto encode = get_encode();
    if (!encode) return cudaErrorNotSupported;
    CUtensorMap tm;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)plan.NT};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = encode(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(x), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    const Layout L(K, N);
    TcParams prm;
    prm.qd = qd;
    prm.scales = scales;
    prm.qzeros = qzeros;
    prm.y = y;
    const size_t tiles = (size_t)plan.NB * plan.MT;
    prm.counters = reinterpret_cast<uint32_t*>(ws);
    prm.partials = ws ? reinterpret_cast<float*>(reinterpret_cast<char*>(ws) + ws_counter_bytes(tiles)) : nullptr;
    prm.M = M;
    prm.N = N;
    prm.K = K;
    prm.G = K / 128;
    prm.NB = plan.NB;
    prm.MT = plan.MT;
    prm.splits = plan.splits;
    const bool pdl = (flags & W4A16_FLAG_PDL) != 0;
    prm.prefetch = pdl && (flags & W4A16_FLAG_STATIC_WEIGHTS) ? 1 : 0;
    switch (plan.NT) {
        case 16: return launch_nt<16>(tm, prm, plan, s, pdl);
        case 32: return launch_nt<32>(tm, prm, plan, s, pdl);
        case 64: return launch_nt<64>(tm, prm, plan, s, pdl);
        default: return launch_nt<128>(tm, prm, plan, s, pdl);
    }
}

int tc_read_status() {
    int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_tc_status, sizeof(int)) != cudaSuccess) return W4A16_ECUDA;
    if (cudaMemcpyToSymbol(g_tc_status, &zero, sizeof(int)) != cudaSuccess) return W4A16_ECUDA;
    return v;
}

}  // namespace w4a16
