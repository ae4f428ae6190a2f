// Canonical <-> device layout of the packed 4-bit weights (integer only).
//
// The re-order is the "grid-preserving packing" step of "Quantize the Target,
// Quantize the Drafter" (pith.science review, "Assumptions & free parameters":
// packing puts weights back onto the frozen per-group grid): every 4-bit code
// keeps its value, only its position changes.  The device layout is defined
// in include/w4a16.h; fused gate/up weights (guH > 0) first put their columns
// in the interleaved order of gu_column (kernels.h).
#include "common.cuh"
#include "kernels.h"

namespace w4a16 {


// Decode a device word index into (column n, canonical word row kw).
__device__ __forceinline__ void decode_dev_word(const Layout& L, size_t d, int& n, int& kw) {
    const size_t tile_words = (size_t)2048 * L.KB;
    const int nb = (int)(d / tile_words);
    const int W = L.width(nb);
    size_t r = d - (size_t)nb * tile_words;
    const int kb = (int)(r / ((size_t)W * 16));
    const int r2 = (int)(r - (size_t)kb * W * 16);
    const int c = r2 / (W * 4);
    const int r3 = r2 - c * W * 4;
    const int t = r3 >> 2;
    const int j = r3 & 3;
    n = 128 * nb + t;
    kw = 16 * kb + 4 * c + j;
}

__global__ void pack_kernel(const uint32_t* __restrict__ q, uint32_t* __restrict__ qd, int K, int N, int guH) {
    const Layout L(K, N);
    const size_t total = (size_t)(K / 8) * N;
    for (size_t d = blockIdx.x * (size_t)blockDim.x + threadIdx.x; d < total; d += (size_t)gridDim.x * blockDim.x) {
        int n, kw;
        decode_dev_word(L, d, n, kw);
        const uint32_t w = q[(size_t)kw * N + (guH ? gu_column(n, guH) : n)];
        uint32_t o = 0;
#pragma unroll
        for (int r = 0; r < 8; ++r) o |= ((w >> (4 * r)) & 0xFu) << (4 * dev_nibble_pos(r));
        qd[d] = o;
    }
}

__global__ void unpack_kernel(const uint32_t* __restrict__ qd, uint32_t* __restrict__ q, int K, int N, int guH) {
    const Layout L(K, N);
    const size_t total = (size_t)(K / 8) * N;
    for (size_t d = blockIdx.x * (size_t)blockDim.x + threadIdx.x; d < total; d += (size_t)gridDim.x * blockDim.x) {
        int n, kw;
        decode_dev_word(L, d, n, kw);
        const uint32_t o = qd[d];
        uint32_t w = 0;
#pragma unroll
        for (int r = 0; r < 8; ++r) w |= ((o >> (4 * dev_nibble_pos(r))) & 0xFu) << (4 * r);
        q[(size_t)kw * N + (guH ? gu_column(n, guH) : n)] = w;
    }
}

static int grid_for(size_t total) {
    size_t b = (total + 255) / 256;
    return (int)(b > 65535 ? 65535 : (b == 0 ? 1 : b));
}

cudaError_t launch_pack(const uint32_t* q, uint32_t* qd, int K, int N, int guH, cudaStream_t s) {
    pack_kernel<<<grid_for((size_t)(K / 8) * N), 256, 0, s>>>(q, qd, K, N, guH);
    return cudaGetLastError();
}

cudaError_t launch_unpack(const uint32_t* qd, uint32_t* q, int K, int N, int guH, cudaStream_t s) {
    unpack_kernel<<<grid_for((size_t)(K / 8) * N), 256, 0, s>>>(qd, q, K, N, guH);
    return cudaGetLastError();
}

}  // namespace w4a16
