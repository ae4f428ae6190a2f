// Sliding-window decode attention on sm_103a: TMA + tcgen05, rows in TMEM lanes.
//
// The drafter's attention restricted to the W most recent keys ("Quantize the
// Target, Quantize the Drafter", pith.science review, "Assumptions & free
// parameters": SWA window 1024 on the leaderboard, 1024 or 2048 after the
// latency / acceptance trade-off; the 16-token DFlash block), for a block of
// nq query tokens appended at the end of a context of L tokens:
//
//     out[i, h] = softmax_{j in J_i}(q[i, h] . k[hk, j] / sqrt(d)) v[hk, j],
//     J_i = [max(0, e_i - W + 1), e_i],  e_i = L - nq + i (causal) or L - 1 (block),
//     hk = h / (Hq / Hkv),  d = 128.
//
// Work: CTA (c, hk) takes the 128 keys [j0 + 128 c, j0 + 128 c + 128) of key /
// value head hk, j0 the block's first visible key rounded down to 8.  Its
// 128 TMEM lanes are the R = nq * Hq / Hkv query rows of the head group (row
// r = query r / G, head hk G + r % G; rows >= R are zero):
//
//   * row threads (warps 0-3, thread r = lane r) put q[r] into TMEM (the A
//     operand of S = Q K^T);
//   * one elected lane of warp 4 loads the key chunk [128 keys][128 d] and the
//     value chunk [128 d][128 keys] (the value cache is kept transposed per
//     head, [d][Lmax], so that both products read K-major operands) with four
//     TMA boxes, then issues the 8 MMAs of S = Q K^T (kind::f16, f32 in TMEM);
//   * row threads read their row of S, mask the keys outside their window,
//     take the row maximum m and p = 2^(s log2(e) / sqrt(d) - m) in f32,
//     l = sum p, and write p as bfloat16 pairs back to TMEM;
//   * warp 4 issues the 8 MMAs of O = P V (A = P from TMEM, B = the value
//     chunk), and the row threads store O, m and l of their row as f32
//     partials;
//   * a second kernel (a programmatic dependent) combines the chunks of every
//     row, out = sum_c 2^(m_c - M) O_c / sum_c 2^(m_c - M) l_c, one CTA per
//     query and head group (a thread per head and column), and writes
//     bfloat16; the partials of a call stay in L2.
//
// Every wait is bounded (common.cuh); on a timeout the kernel records
// W4A16_ETIMEOUT, still drains its tensor-core work, frees its tensor memory
// and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"

namespace w4a16 {

static __device__ int g_swa_status;

struct SwaParams {
    const uint16_t* q;   // [nq][Hq][128] bf16
    uint16_t* out;       // [nq][Hq][128] bf16
    float* part_o;       // [Hkv][C][128][128]
    float* part_ml;      // [Hkv][C][128][2]
    int nq, Hq, Hkv, G, R, L, W, block, j0, C;
};

constexpr int kSwaD = 128;        // head width
constexpr int kSwaKeys = 128;     // keys per CTA
constexpr int kSwaThreads = 160;  // four row warps + the copy / MMA warp
constexpr int kSwaKOff = 0;       // key chunk: two 16 KB slabs (d 0..63, 64..127), [128 keys][128 B]
constexpr int kSwaVOff = 32768;   // value chunk: two 16 KB slabs (keys 0..63, 64..127), [128 d][128 B]
constexpr int kSwaBarOff = 65536;
// Shared memory asked for: the 65 KB the CTA uses, rounded up so that only one
// CTA fits on an SM -- each allocates all 512 tensor-memory columns.
constexpr int kSwaSmem = 116 * 1024;
static_assert(kSwaBarOff + 128 + 1024 <= kSwaSmem, "shared memory layout");
// tensor-memory columns
constexpr uint32_t kSwaTQ = 0, kSwaTS = 64, kSwaTP = 192, kSwaTO = 256;

W4A16_DEVICE void tmem_st_x32s(uint32_t taddr, const uint32_t* v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
        "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
        "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
        "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}

W4A16_DEVICE uint32_t pack_bf16(float lo, float hi) {
    return (uint32_t)f32_to_bf16_rn(lo) | ((uint32_t)f32_to_bf16_rn(hi) << 16);
}

__global__ void __launch_bounds__(kSwaThreads, 1)
    swa_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
               const SwaParams p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem =
        reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kSwaBarOff);
    uint64_t* tma_bar = bars;      // both chunks landed
    uint64_t* q_bar = bars + 1;    // q rows in TMEM (128 row threads)
    uint64_t* s_bar = bars + 2;    // S = Q K^T done
    uint64_t* p_bar = bars + 3;    // P in TMEM (128 row threads)
    uint64_t* o_bar = bars + 4;    // O = P V done
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 5);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.x, hk = blockIdx.y;
    const int key0 = p.j0 + kSwaKeys * c;  // first key of this chunk

    if (threadIdx.x == 0) {
        mbar_init(tma_bar, 1);
        mbar_init(q_bar, 128);
        mbar_init(s_bar, 1);
        mbar_init(p_bar, 128);
        mbar_init(o_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 4) {
        tmem_alloc(tmem_holder, 512);
        tmem_relinquish();
        if (lane == 0) {
            prefetch_tmap(&tmap_k);
            prefetch_tmap(&tmap_v);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    pdl_launch_dependents();
    pdl_wait();  // q and the caches are written by the preceding work

    if (warp == 4) {
        // ------------------------------------------------ copies and MMAs
        if (elect_one()) {
            mbar_arrive_expect_tx(tma_bar, 65536u);
            tma_load_3d(smem + kSwaKOff, &tmap_k, 0, key0, hk, tma_bar);
            tma_load_3d(smem + kSwaKOff + 16384, &tmap_k, 64, key0, hk, tma_bar);
            tma_load_3d(smem + kSwaVOff, &tmap_v, key0, 0, hk, tma_bar);
            tma_load_3d(smem + kSwaVOff + 16384, &tmap_v, key0 + 64, 0, hk, tma_bar);
            bool ok = mbar_wait(q_bar, 0, abort_flag, &g_swa_status) &&
                      mbar_wait(tma_bar, 0, abort_flag, &g_swa_status);
            constexpr uint32_t idesc = idesc_bf16_f32(128, 128);
            if (ok) {
                tc_fence_after();
                const uint32_t kb = smem_u32(smem + kSwaKOff);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16_ts(tmem + kSwaTS, tmem + kSwaTQ + kk * 8,
                                smem_desc_sw128(kb + (kk >> 2) * 16384 + (kk & 3) * 32), idesc, kk > 0 ? 1u : 0u);
            }
            mma_commit(s_bar);  // also after a failed wait, so the row threads' wait ends
            ok = ok && mbar_wait(p_bar, 0, abort_flag, &g_swa_status);
            if (ok) {
                tc_fence_after();
                const uint32_t vb = smem_u32(smem + kSwaVOff);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16_ts(tmem + kSwaTO, tmem + kSwaTP + kk * 8,
                                smem_desc_sw128(vb + (kk >> 2) * 16384 + (kk & 3) * 32), idesc, kk > 0 ? 1u : 0u);
            }
            mma_commit(o_bar);
            if (!ok) *abort_flag = 1;
            // the copies must have landed, and the MMAs finished, before the
            // CTA may free its tensor memory and exit
            (void)mbar_wait(tma_bar, 0, nullptr, &g_swa_status);
            (void)mbar_wait(o_bar, 0, nullptr, &g_swa_status);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------ row threads
        const int r = threadIdx.x;                    // TMEM lane = query row
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        const bool valid = r < p.R;
        const int qi = r / p.G;
        const int rq = valid ? r : 0;  // rows past R read nothing
        // q[r] into TMEM columns 0..63 as bf16 pairs (zero rows beyond R)
        {
            uint32_t v[32];
            const uint4* src = reinterpret_cast<const uint4*>(
                p.q + ((size_t)(rq / p.G) * p.Hq + (size_t)hk * p.G + (rq - (rq / p.G) * p.G)) * kSwaD);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const uint4 w = valid ? __ldg(src + half * 8 + u) : make_uint4(0, 0, 0, 0);
                    v[4 * u] = w.x;
                    v[4 * u + 1] = w.y;
                    v[4 * u + 2] = w.z;
                    v[4 * u + 3] = w.w;
                }
                tmem_st_x32s(tmem + lane_base + kSwaTQ + 32 * half, v);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(q_bar);
        }
        // this row's window, and the scale of the scores in the base-2 exponent
        const int e = p.block ? p.L - 1 : p.L - p.nq + qi;
        const int lo = e - p.W + 1 > 0 ? e - p.W + 1 : 0;
        const float scale = 1.4426950408889634f * rsqrtf((float)kSwaD);
        bool ok = mbar_wait_warp(s_bar, 0, abort_flag, &g_swa_status);
        float m = -INFINITY, l = 0.f;
        if (ok) {
            tc_fence_after();
            // pass 1: the row maximum over the window's keys of this chunk
#pragma unroll 1
            for (int c0 = 0; c0 < kSwaKeys; c0 += 32) {
                uint32_t sv[32];
                tmem_ld_x16(tmem + lane_base + kSwaTS + c0, *reinterpret_cast<uint32_t(*)[16]>(sv));
                tmem_ld_x16(tmem + lane_base + kSwaTS + c0 + 16, *reinterpret_cast<uint32_t(*)[16]>(sv + 16));
                tmem_wait_ld();
#pragma unroll
                for (int u = 0; u < 32; ++u) {
                    const int j = key0 + c0 + u;
                    if (j >= lo && j <= e) m = fmaxf(m, __uint_as_float(sv[u]) * scale);
                }
            }
            // pass 2: p = 2^(s - m), l = sum p over the bf16-rounded p, P into TMEM
#pragma unroll 1
            for (int c0 = 0; c0 < kSwaKeys; c0 += 32) {
                uint32_t sv[32];
                tmem_ld_x16(tmem + lane_base + kSwaTS + c0, *reinterpret_cast<uint32_t(*)[16]>(sv));
                tmem_ld_x16(tmem + lane_base + kSwaTS + c0 + 16, *reinterpret_cast<uint32_t(*)[16]>(sv + 16));
                tmem_wait_ld();
                uint32_t pk[16];
#pragma unroll
                for (int u = 0; u < 32; u += 2) {
                    const int j = key0 + c0 + u;
                    const float p0 = (j >= lo && j <= e) ? exp2f(__uint_as_float(sv[u]) * scale - m) : 0.f;
                    const float p1 = (j + 1 >= lo && j + 1 <= e) ? exp2f(__uint_as_float(sv[u + 1]) * scale - m) : 0.f;
                    pk[u / 2] = pack_bf16(p0, p1);
                    l += bf16lo(pk[u / 2]) + bf16hi(pk[u / 2]);
                }
                tmem_st_x8(tmem + lane_base + kSwaTP + c0 / 2, *reinterpret_cast<const uint32_t(*)[8]>(pk));
                tmem_st_x8(tmem + lane_base + kSwaTP + c0 / 2 + 8, *reinterpret_cast<const uint32_t(*)[8]>(pk + 8));
            }
            tmem_wait_st();
        }
        tc_fence_before();
        mbar_arrive(p_bar);  // also after a failed wait: the MMA lane's wait then ends
        ok = mbar_wait_warp(o_bar, 0, abort_flag, &g_swa_status) && ok;
        if (ok) {
            tc_fence_after();
            float* po = p.part_o + (((size_t)hk * p.C + c) * 128 + r) * kSwaD;
#pragma unroll 1
            for (int c0 = 0; c0 < kSwaD; c0 += 32) {
                uint32_t ov[32];
                tmem_ld_x16(tmem + lane_base + kSwaTO + c0, *reinterpret_cast<uint32_t(*)[16]>(ov));
                tmem_ld_x16(tmem + lane_base + kSwaTO + c0 + 16, *reinterpret_cast<uint32_t(*)[16]>(ov + 16));
                tmem_wait_ld();
                if (valid) {
#pragma unroll
                    for (int u = 0; u < 32; u += 4)
                        *reinterpret_cast<float4*>(po + c0 + u) =
                            make_float4(__uint_as_float(ov[u]), __uint_as_float(ov[u + 1]),
                                        __uint_as_float(ov[u + 2]), __uint_as_float(ov[u + 3]));
                }
            }
            if (valid) {
                float* pml = p.part_ml + (((size_t)hk * p.C + c) * 128 + r) * 2;
                pml[0] = m;
                pml[1] = l;
            }
        }
        if (!ok) *abort_flag = 1;
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 4) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// Combine the chunks of the query rows of one (query, key/value head): CTA
// (qi, hk), thread (hh, t) = column t of head hh of the group (heads hh,
// hh + Gb, ... when the group is wider than the block):
// out = sum_c 2^(m_c - M) O_c[t] / sum_c 2^(m_c - M) l_c, M = max_c m_c.  The
// chunks are read kSwaCB at a time, every load of a batch in flight together
// (one round trip to L2 per batch), and merged with a running maximum: for up
// to kSwaCB chunks (windows up to 1920 keys) the arithmetic is the plain
// formula in chunk order.  Measured: the earlier form (one thread per column,
// the group's heads in turn, the chunks' maximum and then their sums as two
// dependent loops) took ~9 of the 19 us of a 16-token block over 1024 keys.
constexpr int kSwaCB = 16;

__global__ void __launch_bounds__(1024) swa_combine_kernel(const SwaParams p) {
    pdl_wait();  // the partials of the chunk kernel
    const int qi = blockIdx.x, hk = blockIdx.y, t = threadIdx.x & 127;
    const int Gb = (int)blockDim.x >> 7;
    for (int hh = threadIdx.x >> 7; hh < p.G; hh += Gb) {
        const int r = qi * p.G + hh;
        float M = -INFINITY, num = 0.f, den = 0.f;
        for (int c0 = 0; c0 < p.C; c0 += kSwaCB) {
            float mc[kSwaCB], lc[kSwaCB], oc[kSwaCB];
#pragma unroll
            for (int i = 0; i < kSwaCB; ++i) {
                mc[i] = -INFINITY;
                lc[i] = 0.f;
                oc[i] = 0.f;
                if (c0 + i < p.C) {
                    const size_t row = ((size_t)hk * p.C + c0 + i) * 128 + r;
                    mc[i] = __ldcg(p.part_ml + row * 2);
                    lc[i] = __ldcg(p.part_ml + row * 2 + 1);
                    oc[i] = __ldcg(p.part_o + row * kSwaD + t);
                }
            }
            float Mb = M;
#pragma unroll
            for (int i = 0; i < kSwaCB; ++i) Mb = fmaxf(Mb, mc[i]);
            if (c0 > 0) {  // the earlier batches' sums, rescaled to the new maximum
                const float fr = M == -INFINITY ? 0.f : exp2f(M - Mb);
                num *= fr;
                den *= fr;
            }
#pragma unroll
            for (int i = 0; i < kSwaCB; ++i) {
                const float f = mc[i] == -INFINITY ? 0.f : exp2f(mc[i] - Mb);  // no key of this row's window in chunk c
                num = fmaf(f, oc[i], num);
                den = fmaf(f, lc[i], den);
            }
            M = Mb;
        }
        p.out[((size_t)qi * p.Hq + (size_t)hk * p.G + hh) * kSwaD + t] = f32_to_bf16_rn(num / den);
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

static PFN_cuTensorMapEncodeTiled_v12000 swa_encode() {
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

// Workspace: the f32 partials (m and l of every row and chunk, then O) after
// the 64 KB area where the GEMM kernels keep their split-K arrival counters.
// That area is never written here, so one buffer can serve both calls: the
// counters must stay zero between GEMM calls.
static size_t swa_counter_bytes(int) { return kCounterBytes; }

bool swa_plan(int nq, int Hq, int Hkv, int L, int W, int block, SwaPlan* out) {
    const int e0 = block ? L - 1 : L - nq;  // the first query's last visible key
    int lo = e0 - W + 1;
    if (lo < 0) lo = 0;
    const int j0 = lo & ~7;
    const int C = (L - j0 + kSwaKeys - 1) / kSwaKeys;
    out->j0 = j0;
    out->C = C;
    out->G = Hq / Hkv;
    out->R = nq * (Hq / Hkv);
    out->ws_bytes = swa_counter_bytes(Hkv) + (size_t)Hkv * C * 128 * (kSwaD + 2) * sizeof(float);
    return true;
}

cudaError_t launch_swa(const uint16_t* q, const uint16_t* kc, const uint16_t* vtc, uint16_t* out, int nq, int Hq,
                       int Hkv, int L, int Lmax, int W, int block, void* ws, const SwaPlan& plan, cudaStream_t s,
                       bool pdl) {
    auto encode = swa_encode();
    if (!encode) return cudaErrorNotSupported;
    CUtensorMap tk, tv;
    {
        // keys: [Hkv][Lmax][128] viewed as (128 columns, L rows, Hkv heads): rows past L read as zero
        const cuuint64_t dims[3] = {(cuuint64_t)kSwaD, (cuuint64_t)L, (cuuint64_t)Hkv};
        const cuuint64_t strides[2] = {(cuuint64_t)kSwaD * 2, (cuuint64_t)Lmax * kSwaD * 2};
        const cuuint32_t box[3] = {64, (cuuint32_t)kSwaKeys, 1};
        const cuuint32_t estr[3] = {1, 1, 1};
        if (encode(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(kc), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        // values, transposed: [Hkv][128][Lmax] viewed as (L keys, 128 rows, Hkv heads)
        const cuuint64_t dims[3] = {(cuuint64_t)L, (cuuint64_t)kSwaD, (cuuint64_t)Hkv};
        const cuuint64_t strides[2] = {(cuuint64_t)Lmax * 2, (cuuint64_t)kSwaD * Lmax * 2};
        const cuuint32_t box[3] = {64, (cuuint32_t)kSwaD, 1};
        const cuuint32_t estr[3] = {1, 1, 1};
        if (encode(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(vtc), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    SwaParams prm;
    prm.q = q;
    prm.out = out;
    prm.part_ml = reinterpret_cast<float*>(reinterpret_cast<char*>(ws) + swa_counter_bytes(Hkv));
    prm.part_o = prm.part_ml + (size_t)Hkv * plan.C * 128 * 2;
    prm.nq = nq;
    prm.Hq = Hq;
    prm.Hkv = Hkv;
    prm.G = plan.G;
    prm.R = plan.R;
    prm.L = L;
    prm.W = W;
    prm.block = block;
    prm.j0 = plan.j0;
    prm.C = plan.C;
    static int set_for[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!set_for[dev]) {
        e = cudaFuncSetAttribute(swa_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSwaSmem);
        if (e != cudaSuccess) return e;
        set_for[dev] = 1;
    }
    e = launch_kernel(swa_kernel, dim3(plan.C, Hkv), dim3(kSwaThreads), (size_t)kSwaSmem, s, pdl, tk, tv, prm);
    if (e != cudaSuccess) return e;
    const int Gb = plan.G < 8 ? plan.G : 8;  // heads of the group a combine CTA holds at once
    return launch_kernel(swa_combine_kernel, dim3(nq, Hkv), dim3(kSwaD * Gb), 0, s, true, prm);
}

int swa_read_status() {
    int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_swa_status, sizeof(int)) != cudaSuccess) return W4A16_ECUDA;
    if (cudaMemcpyToSymbol(g_swa_status, &zero, sizeof(int)) != cudaSuccess) return W4A16_ECUDA;
    return v;
}

}  // namespace w4a16
