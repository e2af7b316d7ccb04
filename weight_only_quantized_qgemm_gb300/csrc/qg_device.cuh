// Device-side building blocks for the sm_103a kernels: mbarriers with bounded
// waits, TMA bulk / tensor copies with L2 cache hints, tcgen05 (TMEM
// allocation, loads/stores, MMA, commit) and the two register dequantisers.
// Everything is inline PTX; no library code is involved.
#pragma once

#include <cstdint>
#include <cuda.h>

namespace qg {

// ----------------------------------------------------------------- status
// Device status bits (the host maps a non-zero word to a qg_status).
constexpr uint32_t kDevTimeout = 1u;

struct WaitCtl {
    uint64_t timeout_ns;      // per-wait bound
    uint32_t* status;         // global status word
    volatile int* abort;      // CTA-wide abort flag (shared memory)
};

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void raise_abort(const WaitCtl& c, uint32_t code) {
    *c.abort = 1;
    atomicOr(c.status, code);
}

// ----------------------------------------------------------------- smem / mbarrier
// True in exactly one active lane of the (converged) warp.
__device__ __forceinline__ bool elect_one() {
    uint32_t e;
    asm volatile("{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}" : "=r"(e));
    return e != 0;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
        "r"(bytes)
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// As mbar_try_wait, but a thread whose phase is not complete yet sleeps until
// it completes or `ns` nanoseconds pass, instead of polling: polling warps take
// issue slots from the warps doing the work.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity to complete.  Returns false if the
// CTA is aborting or the wait ran past its bound (which starts the abort).
// The iteration cap is a second, clock-independent bound.
static __device__ __noinline__ bool wait_bounded_slow(uint32_t bar, uint32_t parity, const WaitCtl& c) {
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 0; it < (1u << 26); ++it) {
        if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
        if (*c.abort) return false;
        if (globaltimer() - t0 > c.timeout_ns) {
            raise_abort(c, kDevTimeout);
            return false;
        }
    }
    raise_abort(c, kDevTimeout);
    return false;
}

__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const WaitCtl& c) {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_bounded_slow(bar, parity, c);
}

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Programmatic dependent launch: wait for the preceding grid on the stream
// (and its memory) / let the next grid be scheduled.  Both are no-ops for a
// grid launched without the programmatic-serialization attribute.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dependents_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ----------------------------------------------------------------- TMA
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* m) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(m) : "memory");
}

// 2-D tiled tensor copy global -> shared, completion counted on `bar`.
// c0 is the innermost coordinate (elements), c1 the row.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* m, uint32_t bar, int c0,
                                            int c1, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::"
        "cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
        "l"(m), "r"(bar), "r"(c0), "r"(c1), "l"(policy)
        : "memory");
}

// 2-D tiled tensor copy shared -> global (coordinates >= 0, c0 times the
// element size a multiple of 16 bytes); elements outside the tensor are not
// written.  Completion is tracked per thread by bulk groups.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* m, uint32_t src, int c0, int c1) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(m),
                 "r"(src), "r"(c0), "r"(c1)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until at most n of this thread's bulk groups still read shared memory.
template <int n>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(n) : "memory");
}

// Contiguous bulk copy global -> shared (16-byte aligned addresses, size % 16 == 0).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                          uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], "
        "[%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// 16-byte copy global -> shared through the load/store path (not the TMA
// engine), completion tracked per thread by commit groups.  src_bytes = 0
// reads nothing and fills zeros.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Waits until at most n of this thread's committed groups are still pending.
template <int n>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(n) : "memory");
}

// ----------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[tmem] x B[smem]^T, kind::f16 (BF16 or FP16 inputs, FP32 accumulate).
__device__ __forceinline__ void mma_ts_f16(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[smem] x B[smem]^T, kind::f16 (A and B of one type, set by
// the instruction descriptor); both operands through shared-memory
// descriptors.
__device__ __forceinline__ void mma_ss_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[smem] x B[smem]^T, kind::f8f6f4 (E4M3 x E4M3 products, FP32
// accumulate); both operands through shared-memory descriptors.
__device__ __forceinline__ void mma_ss_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every tcgen05 operation issued so far by this thread completes.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Each thread of the warp writes 32 consecutive 32-bit columns of its own lane.
__device__ __forceinline__ void tmem_st_x32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, "
        "%29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

// Each thread of the warp reads 16 consecutive 32-bit columns of its own lane.
__device__ __forceinline__ void tmem_st_x16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_ld_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
        "%12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_ld_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
        "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
        "%30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
          "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
          "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// Generic-proxy shared-memory writes become visible to the async proxy
// (tensor core, TMA) once the writer has executed this fence.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Instruction descriptor of tcgen05.mma kind::f16: FP32 accumulator, A and B
// K-major, M = 128, N = n; ab_bf16 selects BF16 (else FP16) for both A and B.
__host__ __device__ constexpr uint32_t idesc_f16(int n, bool ab_bf16) {
    return (1u << 4)                              // D format: F32
           | ((ab_bf16 ? 1u : 0u) << 7)           // A format
           | ((ab_bf16 ? 1u : 0u) << 10)          // B format
           | (static_cast<uint32_t>(n >> 3) << 17)  // N >> 3
           | (static_cast<uint32_t>(128 >> 4) << 24);  // M >> 4
}

// Instruction descriptor of tcgen05.mma kind::f8f6f4: FP32 accumulator, A and
// B both E4M3 (format code 0) and K-major, M = 128, N = n.
__host__ __device__ constexpr uint32_t idesc_f8_e4m3(int n) {
    return (1u << 4)                              // D format: F32
           | (static_cast<uint32_t>(n >> 3) << 17)  // N >> 3
           | (static_cast<uint32_t>(128 >> 4) << 24);  // M >> 4
}

// Shared-memory matrix descriptor for a K-major operand stored with the
// 128-byte swizzle (8-row x 128-byte atoms, 1024 B apart).  `addr` is the
// shared-space byte address of the first row of the K slice.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);        // start address
    d |= static_cast<uint64_t>(16u >> 4) << 16;                // leading byte offset (unused)
    d |= static_cast<uint64_t>(1024u >> 4) << 32;              // stride byte offset
    d |= static_cast<uint64_t>(1u) << 46;                      // descriptor version
    d |= static_cast<uint64_t>(2u) << 61;                      // 128-byte swizzle
    return d;
}

// ----------------------------------------------------------------- dequantisers
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t f16x2_mul(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// ---- activation split for the E4M3 tensor-core path
// Per-halfword unsigned maximum (used on |x| bit patterns, which order like
// the magnitudes they encode).
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Two BF16 values x0 (low half of xw) and x1, already scaled by a power of
// two so that |x| < 256, become a high and a low E4M3 pair with
//   x = hi + lo / 16
// exactly whenever |x| >= 2^-6 (and to within 2^-14 below that):
//  - x is exact in FP16 (8 significant bits, |x| < 256),
//  - hi = E4M3 round-to-nearest-even of x (4 significant bits),
//  - x - hi is exact in FP16 and, as a multiple of x's BF16 quantum no larger
//    than half of hi's quantum, has at most 3 significant bits; times 16 it is
//    an E4M3 value whenever hi is a normal E4M3 number.
// Low byte of each result = element 0.
__device__ __forceinline__ void split_e4m3x2(uint32_t xw, uint16_t& hi, uint16_t& lo) {
    const float f0 = __uint_as_float(xw << 16);
    const float f1 = __uint_as_float(xw & 0xFFFF0000u);
    uint32_t h2, hh, d;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(h2) : "f"(f1), "f"(f0));
    asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(hi) : "r"(h2));
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(hh) : "h"(hi));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(h2), "r"(hh));
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(d), "r"(0x4C004C00u));   // x 16
    asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(lo) : "r"(d));
}

// Exponent of the activation split of one (row, 128-wide K block): with
// `amax` the bit pattern of the block's largest |x| (sign cleared), 2^e
// brings it into [128, 256): e = 134 - (its biased BF16 exponent).  The cap
// at 126 keeps 2^e and 2^-e normal numbers; a block of zeros and subnormals
// takes e = 126.
__device__ __forceinline__ int split_exponent(uint32_t amax) {
    const int e = 134 - static_cast<int>(amax >> 7);
    return e > 126 ? 126 : e;
}

// BF16x2 {2^e, 2^e} for -126 <= e <= 126 (used to scale two X values at once).
__device__ __forceinline__ uint32_t bf16x2_pow2(int e) {
    const uint32_t pw = static_cast<uint32_t>(e + 127) << 7;
    return pw | (pw << 16);
}

// Per half: the larger magnitude of a and b (the sign bit of the result is the
// XOR of the operands' signs; callers mask it off).
__device__ __forceinline__ uint32_t bf16x2_absmax(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// split_e4m3x2 on two BF16 pairs: x0..x3 (low half of xa first) -> hi and lo
// words of four E4M3 codes each, element 0 in the low byte.
__device__ __forceinline__ void split_e4m3x4(uint32_t xa, uint32_t xb, uint32_t& hi, uint32_t& lo) {
    uint16_t h0, l0, h1, l1;
    split_e4m3x2(xa, h0, l0);
    split_e4m3x2(xb, h1, l1);
    asm("mov.b32 %0, {%1, %2};" : "=r"(hi) : "h"(h0), "h"(h1));
    asm("mov.b32 %0, {%1, %2};" : "=r"(lo) : "h"(l0), "h"(l1));
}

// Byte planes of an 8-entry FP16 table e[0..7] given as four FP16x2 words
// E01 = {e0, e1}, E23, E45, E67: lo0/hi0 hold the low/high bytes of e0..e3,
// lo1/hi1 those of e4..e7, so prmt(lo0, lo1, sel) looks up low bytes by code.
struct LutPlanes {
    uint32_t lo0, lo1, hi0, hi1;
};

__device__ __forceinline__ LutPlanes lut_planes(uint32_t e01, uint32_t e23, uint32_t e45, uint32_t e67) {
    LutPlanes p;
    p.lo0 = prmt(e01, e23, 0x6420u);
    p.hi0 = prmt(e01, e23, 0x7531u);
    p.lo1 = prmt(e45, e67, 0x6420u);
    p.hi1 = prmt(e45, e67, 0x7531u);
    return p;
}

// Eight 3-bit codes, one per nibble of w (nibble i = K offset i) -> four
// FP16x2 words {d0,d1}, {d2,d3}, {d4,d5}, {d6,d7}: eight byte permutes (the
// code word is the permute selector) and a shift of the word's high half,
// done as a high multiply so that it runs on the FMA pipe instead of adding
// to the permutes on the integer pipe.
__device__ __forceinline__ void lut3x8_to_f16(uint32_t w, const LutPlanes& t, uint32_t (&o)[4]) {
    const uint32_t w2 = __umulhi(w, 65536u);
    const uint32_t l0 = prmt(t.lo0, t.lo1, w);
    const uint32_t h0 = prmt(t.hi0, t.hi1, w);
    const uint32_t l1 = prmt(t.lo0, t.lo1, w2);
    const uint32_t h1 = prmt(t.hi0, t.hi1, w2);
    o[0] = prmt(l0, h0, 0x5140u);
    o[1] = prmt(l0, h0, 0x7362u);
    o[2] = prmt(l1, h1, 0x5140u);
    o[3] = prmt(l1, h1, 0x7362u);
}

}  // namespace qg
