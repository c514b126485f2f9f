// ptx.cuh -- inline-PTX building blocks for sm_103a kernels: mbarriers with
// bounded waits, TMA tile loads, and the tcgen05 tensor-memory / MMA
// instructions.  Written from the public PTX ISA descriptions of these
// instructions; every wait gives up after a time limit instead of spinning
// forever, so a kernel whose producer never arrives reports an error and
// returns.
#pragma once

#include <cuda.h>
#include <cstdint>

namespace dfa {
namespace ptx {

// Wall-clock budget of one bounded wait before the kernel gives up.
constexpr uint64_t kWaitLimitNs = 4000000000ull;   // 4 s
// Error codes written to the device error flag.
constexpr int kErrTimeout = 1;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smid() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(r));
    return r;
}

// Per-CTA trace record: SM, start, end, items, then three role counters.
__device__ __forceinline__ void trace_cta(uint64_t* trace, int cap, uint64_t t_start, int items) {
    if (trace && (int)blockIdx.x < cap) {
        uint64_t* r = trace + 8 * blockIdx.x;
        r[0] = smid();
        r[1] = t_start;
        r[2] = globaltimer();
        r[3] = (uint64_t)items;
    }
}
__device__ __forceinline__ void trace_count(uint64_t* trace, int cap, int slot, uint64_t v) {
    if (trace && (int)blockIdx.x < cap) trace[8 * blockIdx.x + slot] = v;
}
// Wait-time slots live in a second table after the `cap` records: 8 uint64
// per CTA, indexed by a role-specific slot number.
__device__ __forceinline__ void trace_wait(uint64_t* trace, int cap, int slot, uint64_t ns) {
    if (trace && (int)blockIdx.x < cap) trace[8 * cap + 8 * blockIdx.x + slot] = ns;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// Arrive without release semantics: the arrival does not wait for this
// thread's earlier global writes and reductions to be performed.  For
// hand-offs that only order TMEM reads (completed by tcgen05.wait::ld) before
// the arrival.
__device__ __forceinline__ void mbar_arrive_relaxed(uint64_t* bar) {
    asm volatile("mbarrier.arrive.relaxed.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits until the phase with the given parity has completed.  Gives up (and
// raises the CTA's abort flag and the device error flag) after kWaitLimitNs,
// or returns false early once another thread of the CTA has aborted.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          int* err) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 15u) == 0) {
            if (*abort_flag) return false;
            if (globaltimer() - t0 > kWaitLimitNs) {
                *abort_flag = 1;
                if (err) atomicExch(err, kErrTimeout);
                return false;
            }
        }
    }
}

// Out-of-line bounded wait (keeps cold wait loops out of the hot code) and
// its traced form, which also adds the SM cycles it spent (including the
// blocking first try_wait) to *acc_cycles: the per-role wait profile of the
// trace facility.  R selects a separate copy of the function: a kernel whose
// warpgroups run under different setmaxnreg budgets needs one copy per
// budget (one out-of-line function cannot be compiled for two budgets).
template <int R = 0>
static __device__ __noinline__ bool mbar_wait_slow(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* err) {
    return mbar_wait(bar, parity, abort_flag, err);
}
template <int R = 0>
static __device__ __noinline__ bool mbar_wait_traced(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* err,
                                              uint64_t* acc_cycles) {
    const uint64_t t0 = clock64();
    const bool ok = mbar_wait(bar, parity, abort_flag, err);
    *acc_cycles += clock64() - t0;
    return ok;
}
// Non-blocking test of a phase (never suspends the thread).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Waits by polling test_wait, never suspending the thread, bounded like
// mbar_wait.  For an MMA-issuing thread whose waits are usually short: a
// suspended try_wait resumes a few hundred cycles after the phase completes,
// which leaves the tensor pipe without queued work (measured on the backward:
// about 5% of its time).  The first test is inline; the polling loop is out of
// line (one copy per register budget R, as for mbar_wait_slow), which keeps the
// issuing thread's code short: 0.7% on the backward against an inline loop.
template <int R = 0>
static __device__ __noinline__ bool mbar_spin_slow(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* err) {
    const uint64_t t0 = globaltimer();
    for (uint32_t i = 1;; ++i) {
        if (mbar_test_wait(bar, parity)) return true;
        if ((i & 63u) == 0) {
            if (*abort_flag) return false;
            if (globaltimer() - t0 > kWaitLimitNs) {
                *abort_flag = 1;
                if (err) atomicExch(err, kErrTimeout);
                return false;
            }
        }
    }
}
template <int R = 0>
__device__ __forceinline__ bool mbar_wait_spin(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* err) {
    if (mbar_test_wait(bar, parity)) return true;
    return mbar_spin_slow<R>(bar, parity, abort_flag, err);
}
// Wait for the MMA issuer: a plain test first (the common case is a phase that
// has already completed, and a potentially-suspending try_wait there leaves the
// tensor pipe idle for hundreds of cycles), then the bounded blocking wait.
template <int R = 0>
__device__ __forceinline__ bool mbar_wait_issuer(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                                 int* err) {
    if (mbar_test_wait(bar, parity)) return true;
    return mbar_wait_slow<R>(bar, parity, abort_flag, err);
}
template <int R = 0>
__device__ __forceinline__ bool mbar_wait_acc(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                              int* err, uint64_t* acc_cycles) {
    if (acc_cycles) return mbar_wait_traced<R>(bar, parity, abort_flag, err, acc_cycles);
    if (mbar_try_wait(bar, parity)) return true;
    return mbar_wait_slow<R>(bar, parity, abort_flag, err);
}

// Bulk (TMA) fp32 reduction of a contiguous shared-memory block into global
// memory: both addresses 16-byte aligned, bytes a multiple of 16.  Tracked by
// the issuing thread's bulk-group; bulk_wait_read() before the source is
// rewritten, bulk_wait_all() before the CTA exits.
__device__ __forceinline__ void bulk_reduce_add_f32(float* gdst, const void* ssrc, uint32_t bytes) {
    asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;" ::"l"(gdst),
                 "r"(smem_u32(ssrc)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Named barrier over `count` threads (a multiple of 32); id 0 is __syncthreads.
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
// Named barrier that also ANDs a flag over the participating threads.
__device__ __forceinline__ bool named_bar_and(uint32_t id, uint32_t count, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %3, 0;\n\t"
        "bar.red.and.pred p, %1, %2, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"(id), "r"(count), "r"((uint32_t)v)
        : "memory");
    return r != 0;
}

// Vector fp32 reduction into global memory: 16 bytes, 16-byte aligned.
__device__ __forceinline__ void red_add_v4(float* p, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

// 4 x 4 transpose inside each quad of lanes (lanes 4q..4q+3): on entry lane
// 4q+j holds x[m] = element (j, m) of its quad's block, on exit lane 4q+m holds
// x[j] = element (j, m).  Four shuffles.
__device__ __forceinline__ void quad_transpose(float (&x)[4], int lane) {
    const bool o1 = lane & 1, o2 = lane & 2;
    float r0 = __shfl_xor_sync(0xffffffffu, o1 ? x[0] : x[1], 1);
    float r1 = __shfl_xor_sync(0xffffffffu, o1 ? x[2] : x[3], 1);
    if (o1) { x[0] = r0; x[2] = r1; } else { x[1] = r0; x[3] = r1; }
    r0 = __shfl_xor_sync(0xffffffffu, o2 ? x[0] : x[2], 2);
    r1 = __shfl_xor_sync(0xffffffffu, o2 ? x[1] : x[3], 2);
    if (o2) { x[0] = r0; x[1] = r1; } else { x[2] = r0; x[3] = r1; }
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
// 4-D tiled load global -> shared, completion counted on `bar` in bytes.
// c0 is the innermost coordinate (elements); it must keep 16-byte alignment.
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* m, uint64_t* bar, int c0, int c1,
                                            int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

// Contiguous (untiled) bulk copy global -> shared; addresses 16-byte aligned,
// size a multiple of 16 bytes.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Makes this thread's generic-proxy shared-memory writes visible to the async
// proxy (tensor-core operand reads).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- tcgen05
// Allocates `ncols` TMEM columns (power of two >= 32); whole warp.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle (the layout TMA writes
// with CU_TENSOR_MAP_SWIZZLE_128B into a 1024-byte aligned buffer).
//   lbo: byte offset between 64-element blocks along M/N (MN-major operands)
//   sbo: byte offset between consecutive 8-row groups
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor for kind::f16 with bf16 A/B and fp32 accumulation.
//   a_mn / b_mn: operand stored M-/N-major (true) or K-major (false).
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn, bool b_mn) {
    return (1u << 4)                      // D format: f32
           | (1u << 7)                    // A format: bf16
           | (1u << 10)                   // B format: bf16
           | ((a_mn ? 1u : 0u) << 15)     // A major-ness
           | ((b_mn ? 1u : 0u) << 16)     // B major-ness
           | ((uint32_t)(N >> 3) << 17)   // N / 8
           | ((uint32_t)(M >> 4) << 24);  // M / 16
}

// A shared-memory matrix descriptor held as its two 32-bit words.  The
// start-address field is the low word's bits 0-13 (address >> 4, below 2^14
// for every shared address under 256 KB), so moving a descriptor within
// shared memory is one 32-bit add on the low word that never carries into the
// high word.  The issuing thread competes for issue slots with the busy warps
// of its SM sub-partition, so each instruction it saves per MMA shows: in a
// stand-alone issue loop beside softmax-like warps, 64-bit descriptor adds ran
// at 71.6 cycles per 128x128x16 MMA and these 32-bit adds at 68.1 (64 alone);
// the backward kernel's 128K pass went from 327 to 316 ms with them.  (The
// forward's issue loop measured slower with them and keeps 64-bit adds.)
struct SDesc {
    uint32_t lo, hi;
};
__device__ __forceinline__ SDesc sdesc_words(uint64_t d) { return SDesc{(uint32_t)d, (uint32_t)(d >> 32)}; }
__device__ __forceinline__ SDesc operator+(SDesc d, uint32_t off) { return SDesc{d.lo + off, d.hi}; }

// D[tmem] (+)= A[smem desc] * B[smem desc]; single thread.
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem desc]; single thread.
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// The same two MMAs with descriptors given as SDesc words.
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, SDesc a, SDesc b, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b64 da, db;\n\t"
        "mov.b64 da, {%1, %2};\n\t"
        "mov.b64 db, {%3, %4};\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, p;\n\t}" ::"r"(d_tmem),
        "r"(a.lo), "r"(a.hi), "r"(b.lo), "r"(b.hi), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, SDesc b, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b64 db;\n\t"
        "mov.b64 db, {%2, %3};\n\t"
        "setp.ne.b32 p, %5, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %4, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "r"(b.lo), "r"(b.hi), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrives once on `bar` when every tcgen05 op issued so far by this thread is done.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns, load and wait in one step so the
// destination registers are never read before they are valid.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}
// Split form of a 16-column load: issue now, wait later.  tmem_wait_ld16x2
// waits for every load this thread issued and ties the two destination arrays
// to the wait, so no use of them can be scheduled before it.
__device__ __forceinline__ void tmem_ld16_async(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_wait_ld16x2(uint32_t (&a)[16], uint32_t (&b)[16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]), "+r"(a[6]), "+r"(a[7]),
                   "+r"(a[8]), "+r"(a[9]), "+r"(a[10]), "+r"(a[11]), "+r"(a[12]), "+r"(a[13]), "+r"(a[14]),
                   "+r"(a[15]), "+r"(b[0]), "+r"(b[1]), "+r"(b[2]), "+r"(b[3]), "+r"(b[4]), "+r"(b[5]), "+r"(b[6]),
                   "+r"(b[7]), "+r"(b[8]), "+r"(b[9]), "+r"(b[10]), "+r"(b[11]), "+r"(b[12]), "+r"(b[13]),
                   "+r"(b[14]), "+r"(b[15])
                 :
                 : "memory");
}
__device__ __forceinline__ void tmem_ld32_async(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_wait_ld32(uint32_t (&r)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                   "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                   "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}
// Two 32-column loads (e.g. S and dP of the same rows) under one wait.
__device__ __forceinline__ void tmem_ld32x2(uint32_t ta, uint32_t tb, uint32_t (&a)[32], uint32_t (&b)[32]) {
    tmem_ld32_async(ta, a);
    tmem_ld32_async(tb, b);
    tmem_wait_ld32(a);
    asm volatile(""
                 : "+r"(b[0]), "+r"(b[1]), "+r"(b[2]), "+r"(b[3]), "+r"(b[4]), "+r"(b[5]), "+r"(b[6]), "+r"(b[7]),
                   "+r"(b[8]), "+r"(b[9]), "+r"(b[10]), "+r"(b[11]), "+r"(b[12]), "+r"(b[13]), "+r"(b[14]),
                   "+r"(b[15]), "+r"(b[16]), "+r"(b[17]), "+r"(b[18]), "+r"(b[19]), "+r"(b[20]), "+r"(b[21]),
                   "+r"(b[22]), "+r"(b[23]), "+r"(b[24]), "+r"(b[25]), "+r"(b[26]), "+r"(b[27]), "+r"(b[28]),
                   "+r"(b[29]), "+r"(b[30]), "+r"(b[31])
                 :
                 : "memory");
}

// 32 lanes x 8 consecutive columns (bf16-packed: 16 values).
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}

// 32 lanes x 16 consecutive columns (used for bf16-packed P: 32 values).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Per-warpgroup register budget change (all four warps of a warpgroup execute
// it).  The block's total stays within what it was launched with.
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// ---------------------------------------------------------------- math
// Hardware base-2 exponential (MUFU), flush-to-zero; ex2(-inf) = 0.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// Two fp32 values -> packed bf16x2 (round to nearest even); `lo` in the low half.
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Two probabilities packed to bf16x2, `lo` = 2^(s0 c + n0) and `hi` =
// 2^(s1 c + n1): both exponents from one two-lane fused multiply-add
// (fma.f32x2, each lane rounded as fmaf), then the hardware exp2 as ex2().
__device__ __forceinline__ uint32_t exp2_pack_bf16(float s0, float s1, float c, float n0, float n1) {
    uint32_t r;
    asm("{\n\t.reg .b64 a, b, d;\n\t.reg .f32 lo, hi;\n\t"
        "mov.b64 a, {%1, %2};\n\t"
        "mov.b64 b, {%3, %3};\n\t"
        "mov.b64 d, {%4, %5};\n\t"
        "fma.rn.f32x2 a, a, b, d;\n\t"
        "mov.b64 {lo, hi}, a;\n\t"
        "ex2.approx.ftz.f32 lo, lo;\n\t"
        "ex2.approx.ftz.f32 hi, hi;\n\t"
        "cvt.rn.bf16x2.f32 %0, hi, lo;\n\t}"
        : "=r"(r)
        : "f"(s0), "f"(s1), "f"(c), "f"(n0), "f"(n1));
    return r;
}

// Two softmax-gradient entries packed to bf16x2, `lo` = p0 (u0 - d0) and
// `hi` = p1 (u1 - d1), with the two-lane fp32 instructions of sm_100 and later
// (sub.f32x2, mul.f32x2): each lane is rounded exactly as the scalar
// subtract and multiply, in half the instructions.
__device__ __forceinline__ uint32_t ds_pack_bf16(float p0, float p1, float u0, float u1, float d0, float d1) {
    uint32_t r;
    asm("{\n\t.reg .b64 a, b, c;\n\t.reg .f32 lo, hi;\n\t"
        "mov.b64 a, {%1, %2};\n\t"
        "mov.b64 b, {%3, %4};\n\t"
        "sub.rn.f32x2 a, a, b;\n\t"
        "mov.b64 c, {%5, %6};\n\t"
        "mul.rn.f32x2 a, a, c;\n\t"
        "mov.b64 {lo, hi}, a;\n\t"
        "cvt.rn.bf16x2.f32 %0, hi, lo;\n\t}"
        : "=r"(r)
        : "f"(u0), "f"(u1), "f"(d0), "f"(d1), "f"(p0), "f"(p1));
    return r;
}

// Byte offset of element (row, col) of a [rows][64] bf16 block stored with the
// 128-byte swizzle: 16-byte chunk index XOR (row mod 8).
__device__ __forceinline__ uint32_t sw128_offset(uint32_t row, uint32_t col) {
    const uint32_t chunk = (col >> 3) ^ (row & 7u);
    return row * 128u + chunk * 16u + (col & 7u) * 2u;
}

}  // namespace ptx
}  // namespace dfa
