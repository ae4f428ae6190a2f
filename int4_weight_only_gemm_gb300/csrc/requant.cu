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
// correctly rounded one, rounded to the nearest integer with ties to even
// (rintf), then z is added and the sum clipped to 0..15.
//
// The quotient is needed only to the nearest integer, so it is first taken as
// q0 = w * RN(1/s): with RN(1/s) = (1/s)(1 + e1) and one more rounding,
// |q0 - w/s| <= (2^-24 + 2^-24 + 2^-48)|w/s|, and the correctly rounded
// quotient Q is within 2^-24 |w/s| of w/s, so |q0 - Q| < 2^-21 max(|q0|, 1).
// Unless a half-integer lies that close to q0, rint(q0) = rint(Q); in that
// rare case (exact ties included) Q itself is computed with __fdiv_rn.
//
// One thread makes four adjacent columns' codes of one 32-row chunk: per row
// it reads the four bf16 values with one 8-byte load (a warp reads a whole
// 256-byte tile row), and it writes the four columns' chunk words -- four
// words each, adjacent in the device layout -- as 64 contiguous bytes.  Four
// columns rather than eight keep the thread's registers down, so more warps
// are resident to cover the load latency (measured 52 us against 66 us for
// the gate_up shape).  The rows are read eight at a time, the next eight
// requested while the current ones are decided: ncu had shown the warps
// waiting on their loads most of the time (52 -> 45 us).  The four passes
// run as a loop, not unrolled (a smaller body for the instruction cache:
// 44.7 -> 44.2 us).
#include "common.cuh"
#include "kernels.h"

namespace w4a16 {

constexpr int kRqCols = 4;                      // columns per thread
constexpr int kRqRowThreads = 128 / kRqCols;      // threads covering a 128-column tile row
constexpr int kRqChunks = 128 / kRqRowThreads;    // 32-row chunks per block

__global__ void __launch_bounds__(128) requant_pack_kernel(const uint16_t* __restrict__ w,
                                                           const uint16_t* __restrict__ scales,
                                                           const uint32_t* __restrict__ qzeros,
                                                           uint32_t* __restrict__ qd, int K, int N) {
    constexpr int C = kRqCols;
    const Layout L(K, N);
    const int nb = blockIdx.x;                                              // column tile
    const int chunk = blockIdx.y * kRqChunks + (int)threadIdx.x / kRqRowThreads;  // 32-row chunk of K
    if (chunk >= 4 * L.KB) return;
    const int kb = chunk >> 2, c = chunk & 3;
    const int W = L.width(nb);
    const int t0 = ((int)threadIdx.x % kRqRowThreads) * C;  // first of this thread's C columns
    if (t0 >= W) return;                                    // W is a multiple of 8
    const int n0 = 128 * nb + t0;
    float s[C], rs[C], z[C];
    {
        const uint2 sv = *reinterpret_cast<const uint2*>(scales + (size_t)kb * N + n0);
        const uint32_t sw[2] = {sv.x, sv.y};
        const uint32_t zw = qzeros[(size_t)kb * (N / 8) + (n0 >> 3)] >> (4 * (n0 & 7));
#pragma unroll
        for (int e = 0; e < C; ++e) {
            s[e] = f16_bits_to_f32((uint16_t)(sw[e >> 1] >> (16 * (e & 1))));
            rs[e] = __frcp_rn(s[e]);
            z[e] = (float)((zw >> (4 * e)) & 0xFu);
        }
    }
    const uint16_t* wp = w + (size_t)(128 * kb + 32 * c) * N + n0;
    uint32_t word[C][4];
#pragma unroll
    for (int e = 0; e < C; ++e)
#pragma unroll
        for (int j = 0; j < 4; ++j) word[e][j] = 0;
    // the chunk's rows eight at a time, the next eight requested while the
    // current ones are decided
    uint2 buf[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) buf[i] = __ldcs(reinterpret_cast<const uint2*>(wp + (size_t)i * N));
#pragma unroll 1
    for (int j = 0; j < 4; ++j) {
        uint2 cur[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) cur[i] = buf[i];
        if (j < 3) {
#pragma unroll
            for (int i = 0; i < 8; ++i) buf[i] = __ldcs(reinterpret_cast<const uint2*>(wp + (size_t)(8 * (j + 1) + i) * N));
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {  // row 8j + i of the chunk
            const uint2 v = cur[i];
            const uint32_t vw[2] = {v.x, v.y};
            const int sh = 4 * dev_nibble_pos(i);
#pragma unroll
            for (int e = 0; e < C; ++e) {
                const float wv = __uint_as_float((e & 1) ? (vw[e >> 1] & 0xFFFF0000u) : (vw[e >> 1] << 16));  // exact
                const float q0 = __fmul_rn(wv, rs[e]);
                float r = rintf(q0);
                // distance from q0 to the nearest half-integer against the bound;
                // a non-finite q0 fails the test and takes the exact path too
                if (!(fabsf(0.5f - fabsf(q0 - r)) > 0x1p-20f * fmaxf(fabsf(q0), 1.f)))
                    r = rintf(__fdiv_rn(wv, s[e]));
                const float q = fminf(fmaxf(r + z[e], 0.f), 15.f);
                word[e][j] |= (uint32_t)q << sh;
            }
        }
    }
    uint4* dst = reinterpret_cast<uint4*>(qd + L.block_word(nb, kb) + ((size_t)c * W + t0) * 4);
#pragma unroll
    for (int e = 0; e < C; ++e) dst[e] = make_uint4(word[e][0], word[e][1], word[e][2], word[e][3]);
}

cudaError_t launch_requant_pack(const uint16_t* w, const uint16_t* scales, const uint32_t* qzeros, uint32_t* qd,
                                int K, int N, cudaStream_t s) {
    const Layout L(K, N);
    requant_pack_kernel<<<dim3(L.NB, (4 * L.KB + kRqChunks - 1) / kRqChunks), 128, 0, s>>>(w, scales, qzeros, qd, K,
                                                                                         N);
    return cudaGetLastError();
}

}  // namespace w4a16
