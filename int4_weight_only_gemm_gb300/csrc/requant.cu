// Grid-preserving re-quantization straight into the device layout (sm_103a).
//
// codes[k][n] = clamp(round(w[k][n] / s[g][n]) + z[g][n], 0, 15), g = k / 128:
// the packing step of "Quantize the Target, Quantize the Drafter"
// (pith.science review, "Assumptions & free parameters": packing rounds the
// updated bf16 weights back onto the frozen per-group scales; referee report
// summary: re-packed onto the same grid, so serving is unchanged).  The scales
// and zero points stay as they are; only the 4-bit codes are new.
//
// The pages give neither the rounding rule nor the precision: the decision is
// taken in IEEE binary32 -- w and s are exact there, the quotient is the
// correctly rounded one (__fdiv_rn), rounded to the nearest integer with ties
// to even (rintf), then z is added and the sum clipped to 0..15.
//
// One thread makes one column's 32 codes of one 32-row chunk: it reads 32
// bf16 values (one per row; the threads of a block read each row's 128
// columns as one contiguous run) and writes the chunk's four device words
// with one 16-byte store (the block writes the chunk's 2 KB contiguously).
#include "common.cuh"
#include "kernels.h"

namespace w4a16 {

__global__ void __launch_bounds__(128) requant_pack_kernel(const uint16_t* __restrict__ w,
                                                           const uint16_t* __restrict__ scales,
                                                           const uint32_t* __restrict__ qzeros,
                                                           uint32_t* __restrict__ qd, int K, int N) {
    const Layout L(K, N);
    const int nb = blockIdx.x;     // column tile
    const int kb = blockIdx.y >> 2;  // 128-row group
    const int c = blockIdx.y & 3;    // 32-row chunk of the group
    const int W = L.width(nb);
    const int t = threadIdx.x;
    if (t >= W) return;
    const int n = 128 * nb + t;
    const float s = f16_bits_to_f32(scales[(size_t)kb * N + n]);
    const float z = (float)((qzeros[(size_t)kb * (N / 8) + (n >> 3)] >> (4 * (n & 7))) & 0xFu);
    const uint16_t* wp = w + (size_t)(128 * kb + 32 * c) * N + n;
    uint32_t word[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t o = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float wv = __uint_as_float((uint32_t)wp[(size_t)(8 * j + i) * N] << 16);  // bf16 -> binary32, exact
            const float r = rintf(__fdiv_rn(wv, s));
            const float v = fminf(fmaxf(r + z, 0.f), 15.f);
            o |= (uint32_t)v << (4 * dev_nibble_pos(i));
        }
        word[j] = o;
    }
    *reinterpret_cast<uint4*>(qd + L.block_word(nb, kb) + ((size_t)c * W + t) * 4) =
        make_uint4(word[0], word[1], word[2], word[3]);
}

cudaError_t launch_requant_pack(const uint16_t* w, const uint16_t* scales, const uint32_t* qzeros, uint32_t* qd,
                                int K, int N, cudaStream_t s) {
    const Layout L(K, N);
    requant_pack_kernel<<<dim3(L.NB, 4 * L.KB), 128, 0, s>>>(w, scales, qzeros, qd, K, N);
    return cudaGetLastError();
}

}  // namespace w4a16
