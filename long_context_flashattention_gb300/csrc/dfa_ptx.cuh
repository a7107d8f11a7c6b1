// dfa_ptx.cuh -- thin inline-PTX wrappers for sm_103a: mbarriers with bounded
// waits, TMA tensor loads, bulk copies, and the tcgen05 tensor-core path
// (TMEM allocation, MMA issue, commit, TMEM load/store, fences).
//
// Descriptor encodings follow the PTX ISA's tcgen05 "shared memory
// descriptor" and "instruction descriptor" tables:
//   smem descriptor: [0,14) start>>4, [16,30) leading byte offset>>4,
//                    [32,46) stride byte offset>>4, [46,48) version = 1,
//                    [49,52) base offset, [61,64) swizzle (2 = 128-byte).
//   instr descriptor (kind::f16): [4,6) D format (1 = f32), [7,10) A format
//                    (1 = bf16), [10,13) B format, [15] A MN-major,
//                    [16] B MN-major, [17,23) N>>3, [24,29) M>>4.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace dfa {

// ---------------------------------------------------------------------------
// status word written by kernels into the caller's workspace
// ---------------------------------------------------------------------------
struct DevStatus {
    int code;   // 0 ok, else a dfa_status value
    int where;  // which wait gave up (role/barrier id)
    int detail; // extra info (iteration, unit)
    int pad;
};

constexpr int kStatusTimeout = 5;  // == DFA_ERR_TIMEOUT
constexpr int kStatusBounds = 6;   // == DFA_ERR_BOUNDS

// Index checks of the bounds-checking build (compiled with DFA_DEBUG_BOUNDS):
// in_bounds(st, ok, site, idx) returns ok; when it is false the first
// violation's site and index are recorded in the status word and the caller
// skips the access.  In the normal build it is the constant true.
#ifdef DFA_DEBUG_BOUNDS
__device__ __noinline__ static bool bounds_fail(DevStatus* st, int site, long long idx)
{
    if (st && atomicCAS(&st->code, 0, kStatusBounds) == 0) {
        st->where = site;
        st->detail = (int)(idx > 0x7fffffffll ? 0x7fffffffll : idx);
    }
    return false;
}
__device__ __forceinline__ bool in_bounds(DevStatus* st, bool ok, int site, long long idx)
{
    return ok ? true : bounds_fail(st, site, idx);
}
#else
__device__ __forceinline__ constexpr bool in_bounds(DevStatus*, bool, int, long long)
{
    return true;
}
#endif

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
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

// Everything a bounded wait needs: a CTA-wide abort flag in shared memory (set
// by the first wait that gives up, so every other role stops too), the
// global status word, and the time limit.
struct WaitCtx {
    volatile uint32_t* abort_flag;
    DevStatus* status;
    uint64_t limit_ns;
};

// Wait until the barrier's phase with the given parity has completed.
// Returns false (and leaves the caller to unwind) when the CTA is aborting or
// the limit passed; the first to time out records `where` in the status word.
static __device__ __forceinline__ bool mbar_wait_slow(uint64_t* bar, uint32_t parity, const WaitCtx& w,
                                            int where)
{
    uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity))
            return true;
        if ((it & 63u) == 0) {
            if (*w.abort_flag)
                return false;
            if (globaltimer_ns() - t0 > w.limit_ns) {
                *w.abort_flag = 1u;
                if (atomicCAS(&w.status->code, 0, kStatusTimeout) == 0) {
                    w.status->where = where;
                    w.status->detail = (int)blockIdx.x;
                }
                __threadfence();
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const WaitCtx& w,
                                          int where)
{
    if (mbar_try_wait(bar, parity))
        return true;
    return mbar_wait_slow(bar, parity, w, where);
}

// ---------------------------------------------------------------------------
// TMA (tensor) loads and bulk copies, completion counted on an mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// 4-byte asynchronous global -> shared copy; src_bytes = 0 stores a zero
// without reading `src` (which must still be a valid address).
__device__ __forceinline__ void cp_async_4(uint32_t dst_smem, const void* src, uint32_t src_bytes)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst_smem), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}

// The barrier's current phase also waits for every cp.async this thread has
// issued so far (the arrival is counted in advance, so the barrier's expected
// count is unchanged).
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t* bar)
{
    asm volatile("cp.async.mbarrier.arrive.shared.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: TMEM allocation, fences, MMA, commit
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrive (once) on bar when every tcgen05 async operation issued so far by
// this thread has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar)
{
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// D(tmem) (+)= A(smem desc) * B(smem desc)^T, bf16 in, fp32 accumulate.
// The MMA reads only shared / tensor memory that the async proxy owns, so the
// asm has no "memory" clobber: it stays ordered against the other volatile
// asm (barrier waits, commits) without forcing the compiler to reload every
// value it holds in memory after each issue, which keeps the single issuing
// thread ahead of the tensor pipe.
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

// D(tmem) (+)= A(tmem) * B(smem desc).  A is M=128 lanes x K, two bf16 per column.
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                       uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn_major,
                                                      bool b_mn_major)
{
    return (1u << 4)                               // D = f32
           | (1u << 7)                             // A = bf16
           | (1u << 10)                            // B = bf16
           | ((a_mn_major ? 1u : 0u) << 15)        // A major
           | ((b_mn_major ? 1u : 0u) << 16)        // B major
           | ((uint32_t)(N >> 3) << 17)            // N
           | ((uint32_t)(M >> 4) << 24);           // M
}

// A descriptor advanced by `bytes` (a multiple of 16) along its start address.
__device__ __forceinline__ uint64_t sdesc_add(uint64_t desc, uint32_t bytes)
{
    return desc + (uint64_t)(bytes >> 4);
}

// Shared-memory matrix descriptor, 128-byte swizzle.  saddr must lie in a
// 1024-byte aligned swizzle pattern (start offsets of 32/64/96 bytes inside a
// row are used to step K within one swizzle atom).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes,
                                                uint32_t sbo_bytes)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Shared-memory matrix descriptor, 32-byte swizzle, K-major rows of exactly
// 32 bytes (one K = 16 slice of bf16): 8-row groups are sbo_bytes apart.
__device__ __forceinline__ uint64_t sdesc_sw32(uint32_t saddr, uint32_t sbo_bytes)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)1 << 16;  // leading byte offset: unused for this layout
    d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)6 << 61;
    return d;
}

// ---------------------------------------------------------------------------
// TMEM <-> registers.  32x32b shape: warp w reaches lanes [32 (w%4), +32);
// thread t of the warp gets lane 32 (w%4) + t, columns [col, col + n).
// Loads are asynchronous: call tmem_ld_wait() and then tmem_reg_fence() on
// the destination registers before reading them.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r)
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* r)
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait()
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Ties the registers to a point after tmem_ld_wait(): the compiler may not
// move their uses above this marker.
__device__ __forceinline__ void tmem_reg_fence16(uint32_t* r)
{
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]));
}

__device__ __forceinline__ void tmem_reg_fence32(uint32_t* r)
{
    tmem_reg_fence16(r);
    tmem_reg_fence16(r + 16);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r)
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r)
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait()
{
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Register rebalancing between warpgroups (all four warps of a warpgroup
// execute the same instruction).  A kernel launched with T threads at R
// registers each may redistribute at most T * R registers in total.
// ---------------------------------------------------------------------------
template <int N>
__device__ __forceinline__ void reg_dealloc()
{
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

template <int N>
__device__ __forceinline__ void reg_alloc()
{
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// ---------------------------------------------------------------------------
// small math helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float fmax3(float a, float b, float c)
{
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ float lg2(float x)
{
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Packed fp32 pairs (Blackwell f32x2 arithmetic): lo in bits [0,32).
__device__ __forceinline__ uint64_t f2pack(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void f2unpack(uint64_t v, float& lo, float& hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ uint64_t f2fma(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ uint64_t f2add(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ uint64_t f2mul(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// two fp32 -> packed bf16x2 (round to nearest even); lo in bits [0,16)
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float bf16lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16hi(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }

// One 16-byte shared-memory store (a single 128-bit access, so that eight
// lanes writing distinct 16-byte columns of a swizzled tile make one
// conflict-free wavefront).
__device__ __forceinline__ void st_shared_v4(uint32_t saddr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(saddr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

// L2 policy that keeps the lines it touches resident ahead of normal lines.
__device__ __forceinline__ uint64_t l2_policy_evict_last()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// *addr += v in L2 (no return value), with an L2 eviction policy.
__device__ __forceinline__ void red_add_f32(float* addr, float v, uint64_t pol)
{
    asm volatile("red.global.add.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(addr), "f"(v), "l"(pol)
                 : "memory");
}

// 128-byte swizzle: byte offset of 16-byte chunk `c` (0..7) of row `r` inside
// a 1024-byte aligned tile whose rows are 128 bytes.
__device__ __forceinline__ uint32_t sw128_offset(uint32_t r, uint32_t c)
{
    return r * 128u + ((c ^ (r & 7u)) << 4);
}

}  // namespace dfa
