/*
 * w4a16.h -- C ABI of the W4A16 group-quantized GEMM library for GB300 (sm_103a).
 *
 *     y[m][n] = sum_k x[m][k] * (q[k][n] - z[k/g][n]) * s[k/g][n]
 *
 * This is the linear layer of the INT4 models in "Quantize the Target,
 * Quantize the Drafter: Efficient Inference with Qwen3.5-4B": an AWQ INT4
 * target whose per-group scales are kept and whose weights are re-packed on
 * the same grid (pith.science review, referee report summary), and a GPTQ
 * INT4 drafter with group size 128 (same review, "Assumptions & free
 * parameters").  Both run it on every decode step and on every verify of a
 * 16-token draft block (DFlash block size 16, same section).
 *
 * The pages give no interface, layout or zero-point convention.  Readings:
 *   - x: bfloat16, row-major [M][K].  y: bfloat16, row-major [M][N], fully
 *     overwritten (no bias, no accumulate), rounded to nearest even.
 *   - qweight (canonical): uint32 [K/8][N]; bits 4i..4i+3 of qweight[j][n]
 *     hold the unsigned 4-bit code of row k = 8j+i.
 *   - scales: IEEE binary16, row-major [K/g][N].
 *   - qzeros: uint32 [K/g][N/8]; bits 4i..4i+3 of qzeros[gi][c] hold the
 *     unsigned 4-bit zero point of column n = 8c+i (packed along N because
 *     K/g is 20 or 76 for some layer shapes, which 8 does not divide).
 *   - weight = (code - zero) * scale, zero used as stored; groups are
 *     contiguous along K (group of row k is k/g).  g = 128 is supported.
 *
 * Device layout (output of w4a16_pack, input of w4a16_gemm): the same
 * K*N/2 bytes, re-ordered into column tiles of 128 (the last tile is
 * W = N - 128*nb wide) and K blocks of 128 rows:
 *   tile nb starts at word 128*16*(K/128)*nb; its block kb at + kb*W*16;
 *   inside a block, word (c*W + t)*4 + j (c, j in 0..3, t < W) holds column
 *   n = 128*nb + t, rows k = 128*kb + 8*(4c + j) + r for r = 0..7;
 *   inside that word, nibble position p holds row offset r = 2p (p < 4) or
 *   r = 2(p-4) + 1 (p >= 4), so that one mask-and-or turns a word shifted by
 *   4p into a bfloat16 pair of rows (2p, 2p+1).
 * A 16-row-by-128-column slab is thus 2 KB contiguous, and a tile's whole K
 * range is contiguous, which is what the kernels stream.
 *
 * Conventions for every call:
 *   - Pointers are DEVICE pointers owned by the caller; the library never
 *     allocates, frees or retains them.  x, y, qweight, qweight_dev,
 *     scales, qzeros and the workspace must be 16-byte aligned.
 *   - Calls are asynchronous on `stream` (0 = legacy default stream); they
 *     return after launching.  Arguments are validated before any launch;
 *     on a non-zero return nothing was launched (W4A16_ECUDA: a launch or a
 *     runtime query failed).  Nothing throws across the ABI.
 *   - y must not overlap any input.  Calls are thread-safe when they use
 *     different workspaces; two calls that may run at the same time on the
 *     GPU must not share one workspace.
 *   - Requirements: M >= 0, N >= 8, N % 8 == 0, K >= 128, K % 128 == 0,
 *     group == 128; M, N, K < 2^31 and K*N/8 < 2^31.  M == 0 (an empty
 *     batch) computes nothing: after the checks of group, N, K (and the
 *     flags) the call returns W4A16_OK without reading any pointer or
 *     launching.
 */
#ifndef W4A16_H
#define W4A16_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; declared opaquely so that this header does not
 * need the CUDA headers. */
typedef struct CUstream_st *w4a16_stream_t;

typedef enum {
    W4A16_OK = 0,
    W4A16_EINVAL = -1,        /* null pointer, bad size, or overlapping output */
    W4A16_EALIGN = -2,        /* a pointer is not 16-byte aligned */
    W4A16_EUNSUPPORTED = -3,  /* group != 128, or K / N outside the supported set */
    W4A16_ECUDA = -4,         /* a CUDA runtime call or kernel launch failed */
    W4A16_ETIMEOUT = -5,      /* a bounded device-side wait gave up (see below) */
    W4A16_EWORKSPACE = -6     /* workspace missing, too small or misaligned */
} w4a16_status;

/*
 * Kernel choice for w4a16_gemm_path.  AUTO looks the problem up in a table
 * generated from times measured on GB300 (every candidate kernel over the
 * decoder's shapes at M = 1 .. 8192), keyed by the weight count K*N (up to
 * 16M, up to 64M, above) and an M bucket: one of the two GEMV forms for small
 * M where it fits, the tensor-core GEMM with the table's token tile otherwise.
 */
typedef enum {
    W4A16_PATH_AUTO = 0,
    W4A16_PATH_GEMV = 1,      /* CUDA-core GEMV, M <= 8: the column-sliced form when the
                                 columns fill the GPU, else the split-K form */
    W4A16_PATH_TC = 2,        /* tcgen05 tensor-core GEMM, any M */
    W4A16_PATH_GEMV_SPLITK = 3, /* CUDA-core GEMV, split-K form forced (M <= 8) */
    W4A16_PATH_GEMV_CS = 4    /* CUDA-core GEMV, column-sliced form forced (M <= 8) */
} w4a16_path;

/*
 * Canonical qweight [K/8][N] -> device layout (same size, documented above).
 * Integer-only and exact; `qweight_dev` must not overlap `qweight`.
 * Grid-preserving packing: codes keep their values, only their order changes
 * (the pages' "re-packs onto the same grid", pith.science review summary).
 */
int w4a16_pack(const uint32_t *qweight, uint32_t *qweight_dev, int K, int N,
               w4a16_stream_t stream);

/* Exact inverse of w4a16_pack: device layout -> canonical [K/8][N]. */
int w4a16_unpack(const uint32_t *qweight_dev, uint32_t *qweight, int K, int N,
                 w4a16_stream_t stream);

/*
 * Grid-preserving re-quantization into the device layout ("Quantize the
 * Target, Quantize the Drafter", pith.science review, "Assumptions & free
 * parameters": packing rounds the updated bf16 weights back onto the frozen
 * per-group scales; referee report summary: re-packed onto the same grid):
 *
 *     code[k][n] = clamp(round(w[k][n] / s[k/128][n]) + z[k/128][n], 0, 15)
 *
 * decided in IEEE binary32: the correctly rounded quotient, rounded to the
 * nearest integer with ties to even, then z added and the sum clipped.  The
 * codes are written in the device layout documented above (the same words
 * w4a16_pack makes from canonical codes), ready for w4a16_gemm with the same
 * scales and qzeros.
 *
 *   w            bf16 [K][N] row-major, device
 *   scales       fp16 [K/group][N], device (the frozen grid)
 *   qzeros       u32 [K/group][N/8], device, nibble n%8 of word n/8
 *   qweight_dev  u32 [K/8][N] words, device, written completely
 *
 * All four 16-byte aligned (W4A16_EALIGN); group must be 128
 * (W4A16_EUNSUPPORTED), K % 128 == 0 and K <= 2 097 024, N % 8 == 0
 * (W4A16_EINVAL / W4A16_EUNSUPPORTED); qweight_dev may not overlap the inputs
 * (W4A16_EINVAL).  Asynchronous on `stream`; the caller owns every buffer.
 * Non-finite w or s give unspecified codes.
 */
int w4a16_requant_pack(const void *w, const void *scales, const uint32_t *qzeros, int K, int N,
                       int group, uint32_t *qweight_dev, w4a16_stream_t stream);

/*
 * Bytes of workspace w4a16_gemm needs for this problem on the current device
 * (0 when the chosen plan needs none).  Returns 0 for invalid arguments too.
 * The workspace carries per-tile arrival counters (its first 64 KB) and
 * split-K partial sums (the rest).  It must be zero-filled once before its
 * first use; every call leaves the counter area at zero again, so one
 * workspace serves any sequence of calls, whatever their shapes.
 */
size_t w4a16_workspace_bytes(int M, int N, int K, int group);

/* Largest workspace any problem with these N, K and M <= max_M can need on
 * the current device. */
size_t w4a16_workspace_bytes_max(int max_M, int N, int K, int group);

/*
 * Registers a caller-owned workspace for the current device, used by
 * w4a16_gemm (NULL, 0 unregisters).  The library keeps only the pointer.
 */
int w4a16_set_workspace(void *workspace, size_t bytes);

/*
 * y = x . dequant(qweight_dev, scales, qzeros), kernel chosen per M.
 * Uses the workspace registered for the current device when the plan needs
 * one (W4A16_EWORKSPACE if it is missing or too small).
 */
int w4a16_gemm(const void *x, const uint32_t *qweight_dev, const void *scales,
               const uint32_t *qzeros, int M, int N, int K, int group, void *y,
               w4a16_stream_t stream);

/* As w4a16_gemm, with an explicit workspace (may be NULL when
 * w4a16_workspace_bytes returns 0). */
int w4a16_gemm_ws(const void *x, const uint32_t *qweight_dev, const void *scales,
                  const uint32_t *qzeros, int M, int N, int K, int group, void *y,
                  void *workspace, size_t workspace_bytes, w4a16_stream_t stream);

/* As w4a16_gemm_ws with an explicit kernel choice (for tests and tuning).
 * W4A16_EUNSUPPORTED when the path cannot run this M. */
int w4a16_gemm_path(int path, const void *x, const uint32_t *qweight_dev,
                    const void *scales, const uint32_t *qzeros, int M, int N, int K,
                    int group, void *y, void *workspace, size_t workspace_bytes,
                    w4a16_stream_t stream);

/* Launch flags for w4a16_gemm_ex. */
enum {
    /* Launch as a programmatic dependent of the preceding work in the stream:
     * the kernel may be scheduled while that work finishes, but reads x, y,
     * the workspace (and, without the next flag, the weights) only after it
     * has completed.  The entry points without a flags argument set it. */
    W4A16_FLAG_PDL = 1u << 0,
    /* With W4A16_FLAG_PDL: the packed weights, scales and zeros are not
     * written by work still in flight on the stream (true for a model whose
     * weights were packed earlier), so the kernel may start streaming them
     * before the preceding work completes. */
    W4A16_FLAG_STATIC_WEIGHTS = 1u << 1,
    /* Tuning: bits 8..15 hold a token-tile width (16, 32, 64, 128 or 192)
     * that the tensor-core kernel uses instead of its dispatch table's choice;
     * 0 keeps the table.  Other values give W4A16_EINVAL.  The split-K
     * workspace depends on the tile: size it with w4a16_workspace_bytes_max. */
    W4A16_FLAG_TOKEN_TILE_SHIFT = 8,
    W4A16_FLAG_TOKEN_TILE_MASK = 0xFFu << 8
};

/* As w4a16_gemm_path with explicit launch flags (W4A16_EINVAL for unknown bits). */
int w4a16_gemm_ex(int path, unsigned flags, const void *x, const uint32_t *qweight_dev,
                  const void *scales, const uint32_t *qzeros, int M, int N, int K, int group,
                  void *y, void *workspace, size_t workspace_bytes, w4a16_stream_t stream);

/*
 * Fused gate/up projection of a gated MLP with its SiLU-multiply epilogue:
 *
 *     y[m][h] = silu(g[m][h]) * u[m][h],   silu(g) = g / (1 + exp(-g)),
 *     g = x . dequant(W[:, h]),  u = x . dequant(W[:, H + h]),  0 <= h < H,
 *
 * for one weight matrix W of [K][2H] whose columns 0..H-1 are the gate
 * projection and H..2H-1 the up projection, quantized with one grid (scales
 * [K/group][2H], zeros [K/group][2H/8], canonical layout as for w4a16_gemm).
 * g and u are accumulated in f32 exactly as w4a16_gemm accumulates y; the
 * epilogue is evaluated in f32 and rounded once to bf16, so the [M][2H]
 * intermediate is never written.
 *
 * The packed weights come from w4a16_pack_gate_up, whose device layout
 * interleaves the halves: in each 128-column tile, per block of 16 columns,
 * 8 gate columns and the 8 matching up columns (a gate column and its up
 * column are then handled by lanes 8 apart of one warp).
 *
 *   x            bf16 [M][K], device;   y   bf16 [M][H], device
 *   qweight_dev  u32 [K/8][2H], device (from w4a16_pack_gate_up)
 *   H            columns of each half: a multiple of 64 (W4A16_EUNSUPPORTED)
 *
 * path, flags, workspace and errors as for w4a16_gemm_ex with N = 2H (the
 * workspace is w4a16_workspace_bytes_path(path, M, 2H, K, group)).
 */
int w4a16_gemm_gate_up_silu(int path, unsigned flags, const void *x, const uint32_t *qweight_dev,
                            const void *scales, const uint32_t *qzeros, int M, int H, int K,
                            int group, void *y, void *workspace, size_t workspace_bytes,
                            w4a16_stream_t stream);

/* Canonical [K/8][2H] fused gate/up codes -> the interleaved device layout of
 * w4a16_gemm_gate_up_silu (same size; H a multiple of 64), and its exact
 * inverse.  Arguments and errors as for w4a16_pack / w4a16_unpack. */
int w4a16_pack_gate_up(const uint32_t *qweight, uint32_t *qweight_dev, int K, int H,
                       w4a16_stream_t stream);
int w4a16_unpack_gate_up(const uint32_t *qweight_dev, uint32_t *qweight, int K, int H,
                         w4a16_stream_t stream);

/* Workspace bytes for a given path (0 if none); 0 for unsupported input. */
size_t w4a16_workspace_bytes_path(int path, int M, int N, int K, int group);

/* The path AUTO takes for this problem on the current device (or < 0). */
int w4a16_auto_path(int M, int N, int K, int group);

/* Static string for a status code. */
const char *w4a16_status_str(int status);

/*
 * Synchronizes `stream`, then returns and clears the device-side status word
 * of the current device: W4A16_OK, or W4A16_ETIMEOUT when a kernel's bounded
 * wait on a barrier gave up (its output is then undefined, the context stays
 * usable).  W4A16_ECUDA if the synchronization itself failed.
 */
int w4a16_last_device_status(w4a16_stream_t stream);

/*
 * Failure-detection self-test.  Launches one thread that waits on a shared-
 * memory barrier which nothing ever completes, through the same bounded wait
 * the GEMM pipelines use, with a limit of `wait_ns` nanoseconds (1e3..1e9).
 * Expected outcome: w4a16_last_device_status(stream) returns W4A16_ETIMEOUT
 * and the context stays usable.  W4A16_EINVAL for a limit out of range.
 */
int w4a16_selftest_wait_timeout(long long wait_ns, w4a16_stream_t stream);

/* Size of the scratch array built into the library for w4a16_gemm_noalloc:
 * 4 MiB, held on every GPU that loads the library until the process exits.
 * The GEMV needs 64 KiB of arrival counters plus 4 KiB of f32 partial sums per
 * CTA at most (one CTA per SM: about 0.7 MiB on a 152-SM GPU), so every
 * M <= 8 problem fits; the size check is a guard, not a limit met in use. */
#define W4A16_NOALLOC_SCRATCH_BYTES (4u << 20)

/*
 * The GEMM for M <= 8 (the split-K GEMV) with no allocation and no workspace
 * argument.  The pages have no counterpart to this call: it exists for callers
 * that may not allocate device memory -- a plugin inside a runtime that plans
 * all device memory itself, code under a locked-down or byte-budgeted
 * allocator -- and so cannot hand the regular entry points the workspace they
 * need for split-K partial sums.  The scratch is instead a fixed array compiled
 * into the library (W4A16_NOALLOC_SCRATCH_BYTES).  The caller still passes x,
 * the packed weights, scales, zeros and y, as for w4a16_gemm.
 *   - Arguments and errors as w4a16_gemm.  M > 8 gives W4A16_EUNSUPPORTED; a
 *     problem whose scratch need exceeds the array gives W4A16_EWORKSPACE.
 *     Nothing is launched then.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture.
 *   - All calls on a device share the array and it keeps the last call's
 *     contents: each call first clears the arrival counters it uses (a memset
 *     on `stream`), and calls that may overlap on the GPU (other streams, other
 *     host threads) race on it, so the caller must serialise them.
 *   - Calls no cudaMalloc, cudaFree or other allocating routine.
 */
int w4a16_gemm_noalloc(const void *x, const uint32_t *qweight_dev, const void *scales,
                       const uint32_t *qzeros, int M, int N, int K, int group, void *y,
                       w4a16_stream_t stream);

/*
 * Sliding-window decode attention of the drafter ("Quantize the Target,
 * Quantize the Drafter", pith.science review, "Assumptions & free
 * parameters": SWA window length 1024 on the leaderboard, 1024 or 2048 after
 * the latency / acceptance trade-off; DFlash block size 16; the gptget.net
 * summary: sliding-window attention reduces long-context decoding latency):
 * a block of nq query tokens at positions L-nq .. L-1 attends, per query head
 * h, to the keys and values of head hk = h / (Hq / Hkv) in its window
 *
 *     J_i = [max(0, e_i - window + 1), e_i],  e_i = L - nq + i (block = 0, causal)
 *                                             e_i = L - 1      (block = 1)
 *     out[i][h] = sum_{j in J_i} softmax_j(q[i][h] . k[hk][j] / sqrt(128)) v[hk][j]
 *
 * with scores and the softmax in f32 (the weights rounded once to bf16 for
 * the tensor-core product with v), the sum in f32, the result rounded to bf16.
 *
 *   q          bf16 [nq][Hq][128], device
 *   k_cache    bf16 [Hkv][Lmax][128], device: row j = key of position j
 *   vt_cache   bf16 [Hkv][128][Lmax], device: the values, transposed per head
 *              (column j = value of position j), so that both products of the
 *              kernel read operands contiguous along their reduction axis
 *   out        bf16 [nq][Hq][128], device, fully written
 *   head_dim   128 (W4A16_EUNSUPPORTED otherwise); Hq % Hkv == 0;
 *              nq * Hq / Hkv <= 128 (W4A16_EUNSUPPORTED); 1 <= nq <= L <= Lmax;
 *              Lmax % 8 == 0; window >= 1; block 0 or 1 (W4A16_EINVAL)
 *   workspace  caller-owned scratch of w4a16_swa_workspace_bytes bytes for the
 *              f32 partial results of the key chunks (W4A16_EWORKSPACE if
 *              missing or short); its first 64 KB are never written, so the
 *              same buffer may also be a GEMM workspace (whose arrival
 *              counters live there).  Two launches: the chunks, then their
 *              combine.
 *   flags      0 or W4A16_FLAG_PDL
 *
 * All pointers 16-byte aligned (W4A16_EALIGN); out may not overlap the
 * inputs (W4A16_EINVAL).  Asynchronous on `stream`; only positions < L of the
 * caches are read.
 */
int w4a16_swa_attention(const void *q, const void *k_cache, const void *vt_cache, int nq, int Hq, int Hkv,
                        int head_dim, int L, int Lmax, int window, int block, void *out, void *workspace,
                        size_t workspace_bytes, unsigned flags, w4a16_stream_t stream);

/* Workspace bytes of w4a16_swa_attention for these sizes (0 for invalid ones). */
size_t w4a16_swa_workspace_bytes(int nq, int Hq, int Hkv, int head_dim, int L, int window, int block);

/* Number of kernel launches the library has issued in this process (every
 * entry point that launches counts its kernel; w4a16_gemm_noalloc's counter
 * memset is not a kernel launch). */
uint64_t w4a16_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* W4A16_H */
