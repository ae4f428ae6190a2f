// Shared device helpers for the W4A16 kernels (sm_103a).
//
// Inline-PTX wrappers for mbarriers, bulk / tensor copies and tcgen05, the
// bounded waits every pipeline uses, and the device-layout arithmetic that
// include/w4a16.h defines.  All waits are bounded: on expiry they record
// W4A16_ETIMEOUT in the translation unit's status word and return false, so a
// lost arrival ends the kernel with an error status instead of a hang.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "w4a16.h"

#define W4A16_DEVICE __device__ __forceinline__

namespace w4a16 {

// ---------------------------------------------------------------------------
// device layout of the packed weights (see the header for the definition)
// ---------------------------------------------------------------------------
struct Layout {
    int K, N, KB, NB;  // KB = K/128 blocks, NB = ceil(N/128) column tiles
    __host__ __device__ Layout(int K_, int N_) : K(K_), N(N_), KB(K_ / 128), NB((N_ + 127) / 128) {}
    __host__ __device__ int width(int nb) const { return N - 128 * nb < 128 ? N - 128 * nb : 128; }
    // word offset of block (nb, kb)
    __host__ __device__ size_t block_word(int nb, int kb) const {
        return (size_t)128 * 16 * KB * nb + (size_t)kb * width(nb) * 16;
    }
};

// position of nibble for row offset r (0..7) inside a device word
__host__ __device__ inline int dev_nibble_pos(int r) { return (r & 1) ? 4 + (r >> 1) : (r >> 1); }

// ---------------------------------------------------------------------------
// time and status
// ---------------------------------------------------------------------------
// Wall-clock bound of any single wait (nanoseconds) and a spin cap.
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint32_t kWaitSpins = 1u << 26;

W4A16_DEVICE uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

W4A16_DEVICE uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

W4A16_DEVICE uint32_t lane_id() {
    uint32_t l;
    asm volatile("mov.u32 %0, %%laneid;" : "=r"(l));
    return l;
}

// ---------------------------------------------------------------------------
// programmatic dependent launch
// ---------------------------------------------------------------------------
// Wait until the grids this one depends on (the preceding work in the stream,
// when launched as a programmatic dependent) have completed and their memory
// is visible.  Returns at once for an ordinary launch.
W4A16_DEVICE void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Let the next programmatic-dependent grid in the stream be scheduled.
W4A16_DEVICE void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
W4A16_DEVICE void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

W4A16_DEVICE void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

W4A16_DEVICE void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

W4A16_DEVICE void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

W4A16_DEVICE void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

W4A16_DEVICE bool mbar_try_wait(uint32_t bar_addr, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar_addr), "r"(parity)
        : "memory");
    return ok != 0;
}

// As mbar_try_wait, but a thread whose phase is not complete sleeps until it
// completes or `ns` nanoseconds pass, instead of returning at once: waiting
// warps then take no issue slots from the working ones.
W4A16_DEVICE bool mbar_try_wait_sleep(uint32_t bar_addr, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar_addr), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}

// Longest single sleep of a bounded wait (the abort flag and the clock are
// checked between sleeps).
constexpr uint32_t kSleepNs = 50000;

// Bounded wait for the phase with the given parity to complete.  `abort` is a
// shared flag: once any thread of the CTA has given up, the others stop
// waiting.  A phase that has already completed costs one poll; otherwise the
// thread sleeps on the barrier between checks of the flag and the clock.
// Returns false on timeout or abort.
W4A16_DEVICE bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort, int* status,
                            uint64_t limit_ns = kWaitNs) {
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait(a, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t i = 0; i < kWaitSpins; ++i) {
        if (abort && *abort) return false;
        if (mbar_try_wait_sleep(a, parity, kSleepNs)) return true;
        if (globaltimer() - t0 > limit_ns) break;
    }
    if (abort) *abort = 1;
    atomicExch(status, (int)W4A16_ETIMEOUT);
    return false;
}

// Warp-uniform bounded wait: every lane waits (so every lane acquires the
// phase), then the warp agrees on the outcome, so the warp-collective tcgen05
// instructions that follow never diverge.
W4A16_DEVICE bool mbar_wait_warp(uint64_t* bar, uint32_t parity, volatile int* abort, int* status) {
    const bool ok = mbar_wait(bar, parity, abort, status);
    return __all_sync(0xFFFFFFFFu, ok) != 0;
}

// One lane of a converged warp is elected (the same lane for every caller).
W4A16_DEVICE bool elect_one() {
    uint32_t pred = 0;
    asm volatile(
        "{\n\t.reg .b32 rx;\n\t.reg .pred px;\n\t"
        "elect.sync rx|px, %1;\n\t"
        "selp.b32 %0, 1, 0, px;\n\t}"
        : "=r"(pred)
        : "r"(0xFFFFFFFFu));
    return pred != 0;
}

// AND of `pred` over the `count` threads of named barrier `id` (all must arrive).
W4A16_DEVICE bool bar_and(int id, int count, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// explicit shared-memory loads (32-bit shared addresses)
// Division by a divisor d >= 1 fixed for the launch, for numerators
// 0 <= n < 2^31, by one multiply-high and a shift (Granlund and Montgomery,
// "Division by invariant integers using multiplication", 1994, theorem 4.2
// with N = 31): with l = ceil(log2 d) and m = ceil(2^(31 + l) / d), which is
// below 2^32, floor(n / d) = floor(m n / 2^(31 + l)).  m = 0 stands for d = 1.
struct FastDiv {
    uint32_t m;
    int s;  // l - 1
};
static inline FastDiv fast_div(int d) {
    FastDiv f{0u, 0};
    if (d <= 1) return f;
    int l = 0;
    while ((1ll << l) < d) ++l;
    f.m = (uint32_t)(((1ull << (31 + l)) + (unsigned long long)d - 1) / (unsigned long long)d);
    f.s = l - 1;
    return f;
}
W4A16_DEVICE int div_by(int n, uint32_t m, int s) { return m ? (int)(__umulhi((uint32_t)n, m) >> s) : n; }

W4A16_DEVICE void sts_u16(uint32_t addr, uint16_t v) {
    asm volatile("st.shared.b16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}
W4A16_DEVICE uint4 lds_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}
W4A16_DEVICE uint32_t lds_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}
W4A16_DEVICE unsigned short lds_u16(uint32_t addr) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
    return v;
}

// ---------------------------------------------------------------------------
// bulk and tensor copies (TMA), global -> shared, completion on an mbarrier
// ---------------------------------------------------------------------------
W4A16_DEVICE void bulk_g2s(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(smem_dst)),
        "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

W4A16_DEVICE void tma_load_2d(void* smem_dst, const void* tmap, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_u32(smem_dst)),
        "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// 4-byte asynchronous copy global -> shared (completion tracked below)
W4A16_DEVICE void cp_async_4(void* smem_dst, const void* gsrc) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(smem_dst)), "l"(gsrc) : "memory");
}
// 8- and 16-byte asynchronous copies global -> shared (both addresses aligned
// to the size); the 16-byte form bypasses L1.
W4A16_DEVICE void cp_async_8(void* smem_dst, const void* gsrc) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(smem_dst)), "l"(gsrc) : "memory");
}
W4A16_DEVICE void cp_async_16(void* smem_dst, const void* gsrc) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gsrc) : "memory");
}
// Close the group of this thread's cp.async copies issued since the last commit.
W4A16_DEVICE void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Wait until at most N of this thread's committed cp.async groups are pending.
template <int N>
W4A16_DEVICE void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// The mbarrier's current phase also waits for this thread's earlier cp.async
// copies (net-zero change to the arrival count).
W4A16_DEVICE void cp_async_mbar_arrive(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.shared.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

W4A16_DEVICE void tma_load_3d(void* smem_dst, const void* tmap, int x, int y, int z, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(smem_u32(smem_dst)),
        "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

W4A16_DEVICE void prefetch_tmap(const void* tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}
W4A16_DEVICE void named_bar(int id, int count) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory"); }

// ---------------------------------------------------------------------------
// tcgen05 (tensor memory and 5th-generation MMA)
// ---------------------------------------------------------------------------
W4A16_DEVICE void tmem_alloc(uint32_t* smem_result, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_result)),
                 "r"(ncols)
                 : "memory");
}
W4A16_DEVICE void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
W4A16_DEVICE void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
W4A16_DEVICE void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
W4A16_DEVICE void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[tmem] * B[smem desc], kind::f16 (bf16 inputs, f32 accumulate)
W4A16_DEVICE void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                              uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// arrive on the mbarrier once all earlier tcgen05 async ops of this thread are done
W4A16_DEVICE void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// The same two, called by all 32 lanes of a converged warp: one lane, chosen
// by elect.sync (the lowest active lane, so the same lane issues and commits),
// executes the instruction.  The operands are computed by the whole warp.
// Measured on GB300 (M = 128, N = 16, K = 16, A in tensor memory): a loop
// run this way issues one MMA every ~8.8 ns; the same loop run by one lane
// alone, inside a branch, one every ~23 ns.
W4A16_DEVICE void mma_bf16_ts_warp(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                   uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

W4A16_DEVICE void mma_commit_warp(uint64_t* bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_u32(bar))
        : "memory");
}

// 32 lanes x 32 bits, 8 consecutive columns per thread
W4A16_DEVICE void tmem_st_x8(uint32_t taddr, const uint32_t (&v)[8]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr), "r"(v[0]),
        "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
        : "memory");
}
W4A16_DEVICE void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

W4A16_DEVICE void tmem_ld_x16(uint32_t taddr, uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr)
        : "memory");
}
W4A16_DEVICE void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes, 8-row groups 1024 bytes apart.  `addr` must keep the 1024-byte
// alignment of the swizzle atom except for the K offset inside the row.
W4A16_DEVICE uint64_t smem_desc_sw128(uint32_t addr) {
    uint64_t d = 0;
    d |= (uint64_t)((addr & 0x3FFFF) >> 4);          // start address
    d |= (uint64_t)(16 >> 4) << 16;                  // leading byte offset (unused here)
    d |= (uint64_t)(1024 >> 4) << 32;                // stride byte offset: next 8 rows
    d |= (uint64_t)1 << 46;                          // descriptor version
    d |= (uint64_t)2 << 61;                          // 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f16: bf16 A and B, f32 D, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ---------------------------------------------------------------------------
// numeric helpers
// ---------------------------------------------------------------------------
// bfloat16 pair (128 + code_lo, 128 + code_hi) from the nibbles at bit 4p and
// bit 4p + 16 of a device word: an exact integer-to-bfloat16 conversion.
W4A16_DEVICE uint32_t magic_pair(uint32_t w, int p) {
    uint32_t r;
    const uint32_t s = w >> (4 * p);
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(s), "r"(0x000F000Fu), "r"(0x43004300u));
    return r;  // (s & 0x000F000F) | 0x43004300
}

W4A16_DEVICE float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
W4A16_DEVICE float bf16hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// d = a.lo * b.lo + c  /  a.hi * b.hi + c  with bf16 inputs, f32 accumulate
W4A16_DEVICE float fma_lo(uint32_t a, uint32_t b, float c) {
    float d;
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
        "mov.b32 {al, ah}, %1;\n\t"
        "mov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.bf16 %0, al, bl, %3;\n\t}"
        : "=f"(d)
        : "r"(a), "r"(b), "f"(c));
    return d;
}
W4A16_DEVICE float fma_hi(uint32_t a, uint32_t b, float c) {
    float d;
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
        "mov.b32 {al, ah}, %1;\n\t"
        "mov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.bf16 %0, ah, bh, %3;\n\t}"
        : "=f"(d)
        : "r"(a), "r"(b), "f"(c));
    return d;
}

W4A16_DEVICE uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
W4A16_DEVICE uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

W4A16_DEVICE uint16_t f32_to_bf16_rn(float f) {
    uint16_t r;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(f));
    return r;
}

W4A16_DEVICE float f16_bits_to_f32(uint16_t h) {
    float f;
    asm("{\n\t.reg .f16 t;\n\tmov.b16 t, %1;\n\tcvt.f32.f16 %0, t;\n\t}" : "=f"(f) : "h"(h));
    return f;
}

// ---------------------------------------------------------------------------
// split-K fix-up: ordered reduction of partial tiles by the last arrival
// ---------------------------------------------------------------------------
// Workspace layout shared by the kernels: a fixed 64 KB area of per-tile
// arrival counters (uint32), then the partial sums (float).  The counter area
// has the same place and size for every problem, so partial sums of one call
// never land where another call keeps its counters; each counter returns to
// zero after its tile's last contributor reduced it.
constexpr size_t kCounterBytes = 64 * 1024;
constexpr size_t kMaxCounters = kCounterBytes / 4;
__host__ __device__ inline size_t ws_counter_bytes(size_t) { return kCounterBytes; }

}  // namespace w4a16
