// Internal interface between the C ABI layer and the kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "w4a16.h"

namespace w4a16 {

// Fused gate/up weights [K][2H] (gate columns 0..H-1, up columns H..2H-1) in
// the device layout: column j of 128-column device tile t holds gate column
// 64t + 8b + r when j % 16 < 8 and up column H + 64t + 8b + r otherwise
// (b = j / 16, r = j % 8), so a gate column and its up column sit 8 apart in
// one warp.  Returns the canonical column of device column n.
__host__ __device__ inline int gu_column(int n, int H) {
    const int t = n >> 7, j = n & 127;
    return ((j & 8) ? H : 0) + 64 * t + 8 * (j >> 4) + (j & 7);
}

// silu(g) * u = g u / (1 + e^-g) in f32, with the fast exponential and
// division (relative error ~1e-6, far below the bf16 rounding of the result;
// e^-g = inf for g < -88 gives 0)
__device__ __forceinline__ float silu_mul(float g, float u) { return __fdividef(g * u, 1.f + __expf(-g)); }

// Argument checks of the GEMM entry points (api.cu): W4A16_OK, or the status
// to return without launching.  ny = columns of y (N, or H for fused gate/up).
int check_gemm(const void* x, const uint32_t* qd, const void* scales, const uint32_t* qzeros, int M, int N, int K,
               int group, void* y, int ny);
// Counts one kernel launch in w4a16_launch_count (api.cu).
void note_launch();

// The dispatch table's row for this problem (api.cu; dispatch_table.h):
// path is W4A16_PATH_GEMV_SPLITK, W4A16_PATH_GEMV_CS or W4A16_PATH_TC, nt the
// tensor-core token tile (0 for the GEMV).
struct DispatchRow;
const DispatchRow* dispatch_row(int M, int K, int N);
int dispatch_nt(int M, int K, int N);  // the table's token tile when it picks the tensor cores, else 0

// guH = 0: plain layout; guH = H: fused gate/up weights with N = 2H columns
cudaError_t launch_pack(const uint32_t* q, uint32_t* qd, int K, int N, int guH, cudaStream_t s);
cudaError_t launch_unpack(const uint32_t* qd, uint32_t* q, int K, int N, int guH, cudaStream_t s);
cudaError_t launch_requant_pack(const uint16_t* w, const uint16_t* scales, const uint32_t* qzeros, uint32_t* qd,
                                int K, int N, cudaStream_t s);

// CUDA-core split-K GEMV (M <= 8)
struct GemvPlan {
    int ctas, P;     // CTAs, range owners (one per CTA)
    int S;           // shared-memory ring stages
    int split, base, extra;  // unit partition (see gemv.cu)
    long long C;     // units: one 128-row group of one 128-column tile
    size_t smem, ws_bytes;
};
bool gemv_plan(int M, int N, int K, int sms, GemvPlan* out);
// guH > 0: fused gate/up weights (N = 2 guH), y is [M][guH] = silu(gate) * up
cudaError_t launch_gemv(const uint16_t* x, const uint32_t* qd, const uint16_t* scales, const uint32_t* qzeros,
                        uint16_t* y, int M, int N, int K, void* ws, const GemvPlan& plan, cudaStream_t s,
                        unsigned flags, int guH);
int gemv_read_status();

// Column-sliced CUDA-core GEMV (M <= 8): every CTA owns whole columns, no workspace
struct GemvCsPlan {
    int ctas;        // one per SM (fewer when the columns are fewer)
    int U, unit;     // column units and their width
    int D;           // ring slots in flight a thread
    int ips;         // items a slot (2 with D = 4, 1 with D = 8 or 4)
    size_t smem;
};
bool gemv_cs_plan(int M, int N, int K, int sms, int guH, GemvCsPlan* out);
cudaError_t launch_gemv_cs(const uint16_t* x, const uint32_t* qd, const uint16_t* scales, const uint32_t* qzeros,
                           uint16_t* y, int M, int N, int K, const GemvCsPlan& plan, cudaStream_t s, unsigned flags,
                           int guH);

// tcgen05 tensor-core GEMM (any M)
struct TcPlan {
    int NT, MT, NB;          // tokens per tile, token tiles, column tiles
    int whole, splits;       // tiles [0, whole) whole, the rest in `splits` K pieces each
    int units;               // whole + (NB * MT - whole) * splits
    int ctas;                // persistent CTAs
    size_t smem, ws_bytes;
};
// force_nt: a token tile (16, 32, 64, 128 or 192) in place of the table's, 0 = the table's
bool tc_plan(int M, int N, int K, int sms, TcPlan* out, int force_nt = 0);
cudaError_t launch_tc(const uint16_t* x, const uint32_t* qd, const uint16_t* scales, const uint32_t* qzeros,
                      uint16_t* y, int M, int N, int K, void* ws, const TcPlan& plan, cudaStream_t s,
                      unsigned flags, int guH);

// Launch `kern` with an optional programmatic-stream-serialization attribute
// and, for cluster > 1, clusters of `cluster` CTAs along x.
template <typename Kern, typename... Args>
cudaError_t launch_kernel_ex(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl, int cluster,
                             Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (cluster > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = (unsigned)cluster;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = n ? attr : nullptr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <typename Kern, typename... Args>
cudaError_t launch_kernel(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl, Args... args) {
    return launch_kernel_ex(kern, grid, block, smem, s, pdl, 0, args...);
}
int tc_read_status();

// sliding-window decode attention (head width 128)
struct SwaPlan {
    int j0, C;       // first key (a multiple of 8) and 128-key chunks of the block's window
    int G, R;        // query heads per key / value head; query rows per head group (nq G)
    size_t ws_bytes;  // the f32 partials
};
bool swa_plan(int nq, int Hq, int Hkv, int L, int W, int block, SwaPlan* out);
cudaError_t launch_swa(const uint16_t* q, const uint16_t* kc, const uint16_t* vtc, uint16_t* out, int nq, int Hq,
                       int Hkv, int L, int Lmax, int W, int block, void* ws, const SwaPlan& plan, cudaStream_t s,
                       bool pdl);
int swa_read_status();

// failure-detection self-test
cudaError_t launch_selftest_wait(uint64_t limit_ns, cudaStream_t s);
int selftest_read_status();

}  // namespace w4a16
