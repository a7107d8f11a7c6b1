// dfa_fwd.cu -- exact attention forward on tcgen05 tensor cores (sm_103a).
//
// Method (FlashAttention glossary entry; Striped Attention Guide,
// "Incremental Online Softmax Rescaling" and "Intra-Block vs. Inter-Block
// Masking Logic"): for a block of query rows keep a running row maximum m,
// running sum l and unnormalised output O; for each key/value tile compute
// S = Q K^T, mask keys whose global position exceeds the query's, rescale
// (l, O) when m grows, add exp(S - m) to l and exp(S - m) V to O; finally
// O / l and LSE = m * scale + ln l.  Fully masked tiles are never visited;
// tiles entirely in the past need no mask.
//
// GB300 mapping (one persistent CTA per SM, 384 threads = 3 warpgroups;
// warps 10-11 only give their registers to the math warpgroups):
//   warp 9      TMA producer: Q tiles (2 x 128 rows) per unit, K/V tiles
//               (128 rows) through a KS-stage ring, 128-byte swizzle.
//   warp 8      MMA issuer (one thread): S_t = Q_t K^T into TMEM (fp32),
//               O_t += P_t V with P_t read from TMEM (bf16, aliased on S_t).
//   warps 0-3   softmax for query tile 0, warps 4-7 for tile 1: one thread
//               per query row (TMEM lane), row max / mask / exp2 / row sum,
//               P written back to TMEM, O rescaled in TMEM only when the
//               running max grows by more than 2^8 (lazy rescale), epilogue.
// TMEM: S0 [0,128) S1 [128,256) O0 [256,256+d) O1 [256+d,256+2d) columns.
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "dfa_params.h"
#include "dfa_ptx.cuh"

namespace dfa {

namespace fwd {

constexpr int kThreads = 384;      // three warpgroups
// Launch: 384 threads x 168 registers = 64512.  The producer/MMA warpgroup
// drops to 120, the two math warpgroups rise to 192: 128 * (192 + 192 + 120)
// = 64512, the launch's total.
constexpr int kRegsMath = 192;
constexpr int kRegsCtl = 120;
static_assert(2 * kRegsMath + kRegsCtl == 3 * 168, "register budget");
constexpr int kRowsPerUnit = 256;  // two 128-row query tiles
constexpr float kRescaleLog2 = 8.0f;

template <int D>
struct Cfg {
    static constexpr int kTile = 128 * D * 2;          // bytes of a 128-row bf16 tile
    static constexpr int kStages = (D == 128) ? 2 : 3;  // K and V ring depth
    static constexpr int kQ0 = 0;
    static constexpr int kK0 = 2 * kTile;
    static constexpr int kV0 = kK0 + kStages * kTile;
    static constexpr int kBar = kV0 + kStages * kTile;
    // barrier indices
    static constexpr int QFULL = 0, QEMPTY = 1, KFULL = 2, KEMPTY = 2 + kStages,
                         VFULL = 2 + 2 * kStages, VEMPTY = 2 + 3 * kStages,
                         SFULL = 2 + 4 * kStages, PFULL = SFULL + 2, OFULL = PFULL + 2,
                         NBAR = OFULL + 2;
    static constexpr int kSmem = kBar + NBAR * 8 + 16 + 1024;  // + tmem slot, flag, align
};

// Per-(unit, kv-chunk step) tiles: visible tiles [j0, jv), of which
// [jf0, jf) need no mask.  A row at position x sees the keys at positions
// [doc_lo(x), causal ? x : doc_hi(x) - 1] (its document; everything without
// documents), an interval of each key chunk because positions increase along
// a chunk.  Union over the unit's rows: [doc_lo(x_min), upper(x_max)];
// intersection: [doc_lo(x_max), upper(x_min)].
// Step s visits key chunk s: every unit takes the chunks in the same order
// (not rotated by its own chunk as a ring of workers would), so the units
// running at one time read the same chunk's K/V tiles out of L2.
struct StepTiles {
    int32_t c, j0, jv, jf0, jf;
};

__device__ __forceinline__ StepTiles step_tiles(const FwdParams& p, const Unit& un, int s)
{
    StepTiles r;
    r.c = s;
    const DevMap& km = p.kmap[r.c];
    if (!p.causal && p.ndocs == 0) {
        r.j0 = 0;
        r.jf0 = 0;
        r.jv = ceil_div(p.chunk_k, 128);
        r.jf = p.chunk_k / 128;
        return r;
    }
    const DevMap& qm = p.qmap[un.chunk];
    const int32_t pq_min = map_pos(qm, un.row0);
    const int32_t pq_max = map_pos(qm, un.row0 + un.nvalid - 1);
    int32_t lo_min, hi_min, lo_max, hi_max;
    doc_range(p.docs, p.ndocs, pq_min, lo_min, hi_min);
    doc_range(p.docs, p.ndocs, pq_max, lo_max, hi_max);
    const int32_t up_max = p.causal ? pq_max : hi_max - 1;
    const int32_t up_min = p.causal ? pq_min : hi_min - 1;
    r.j0 = map_count_le(km, lo_min - 1) / 128;
    r.jv = ceil_div(map_count_le(km, up_max), 128);
    r.jf0 = ceil_div(map_count_le(km, lo_max - 1), 128);
    r.jf = map_count_le(km, up_min) / 128;
    return r;
}

__device__ __forceinline__ int32_t unit_tiles(const FwdParams& p, const Unit& un)
{
    int32_t t = 0;
    for (int s = 0; s < p.nkv; ++s) {
        const StepTiles st = step_tiles(p, un, s);
        t += st.jv > st.j0 ? st.jv - st.j0 : 0;
    }
    return t;
}

// S = Q K^T for one 128-row query tile (D/16 K steps of 16).
template <int D>
__device__ __forceinline__ void issue_s(uint32_t tS, uint64_t dQ0, uint64_t dK0, uint32_t qoff,
                                        uint32_t koff)
{
    constexpr uint32_t idS = idesc_bf16_f32(128, 128, false, false);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
        mma_ss(tS, sdesc_add(dQ0, qoff + off), sdesc_add(dK0, koff + off), idS, kk > 0);
    }
}

// O += P V with P (bf16) in TMEM over the S columns, V MN-major in SMEM.
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t tO, uint32_t tP, uint64_t dV0, uint32_t voff,
                                         bool acc)
{
    constexpr uint32_t idO = idesc_bf16_f32(128, D, false, true);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
        mma_ts(tO, tP + kk * 8, sdesc_add(dV0, voff + kk * 2048), idO, (acc || kk > 0) ? 1u : 0u);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                    const __grid_constant__ CUtensorMap tmv, const __grid_constant__ FwdParams p)
{
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t* bar = (uint64_t*)(smem + C::kBar);
    uint32_t* tmem_slot = (uint32_t*)(bar + C::NBAR);
    volatile uint32_t* abort_flag = tmem_slot + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    WaitCtx wctx{abort_flag, p.status, p.timeout_ns};

    if (threadIdx.x == 0) {
        *abort_flag = 0u;
        mbar_init(&bar[C::QFULL], 1);
        mbar_init(&bar[C::QEMPTY], 1);
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&bar[C::KFULL + s], 1);
            mbar_init(&bar[C::KEMPTY + s], 1);
            mbar_init(&bar[C::VFULL + s], 1);
            mbar_init(&bar[C::VEMPTY + s], 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(&bar[C::SFULL + t], 1);
            mbar_init(&bar[C::PFULL + t], 128);
            mbar_init(&bar[C::OFULL + t], 1);
        }
        fence_barrier_init();
    }
    if (warp == 8) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp >= 8) {
        reg_dealloc<kRegsCtl>();
        if (warp == 9) {
            // ------------------------------------------------------------- producer
            if (lane == 0) {
                prefetch_tmap(&tmq);
                prefetch_tmap(&tmk);
                prefetch_tmap(&tmv);
                uint32_t kc = 0, qc = 0;
                for (int u = blockIdx.x; u < p.total_units; u += gridDim.x) {
                    Unit un = decode_unit(p.units, p.BH, kRowsPerUnit, u, false);
                    if (unit_tiles(p, un) == 0)
                        continue;
                    const int b = un.slice / p.Hq, h = un.slice % p.Hq;
                    const int zk = b * p.Hkv + h / p.G;
                    if (qc > 0 && !mbar_wait(&bar[C::QEMPTY], (qc - 1) & 1, wctx, 10))
                        goto producer_done;
                    mbar_arrive_expect_tx(&bar[C::QFULL], 2 * C::kTile);
                    {
                        const int qrow = un.chunk * p.chunk_q + un.row0;
#pragma unroll
                        for (int t = 0; t < 2; ++t)
#pragma unroll
                            for (int hb = 0; hb < D / 64; ++hb)
                                tma_load_3d(smem + C::kQ0 + t * C::kTile + hb * 16384, &tmq,
                                            &bar[C::QFULL], hb * 64, qrow + t * 128, un.slice);
                    }
                    ++qc;
                    for (int s = 0; s < p.nkv; ++s) {
                        StepTiles st = step_tiles(p, un, s);
                        for (int j = st.j0; j < st.jv; ++j) {
                            const int ks = kc % C::kStages;
                            const uint32_t n = kc / C::kStages;
                            const int krow = st.c * p.chunk_k + j * 128;
                            if (kc >= (uint32_t)C::kStages &&
                                !mbar_wait(&bar[C::KEMPTY + ks], (n - 1) & 1, wctx, 11))
                                goto producer_done;
                            mbar_arrive_expect_tx(&bar[C::KFULL + ks], C::kTile);
#pragma unroll
                            for (int hb = 0; hb < D / 64; ++hb)
                                tma_load_3d(smem + C::kK0 + ks * C::kTile + hb * 16384, &tmk,
                                            &bar[C::KFULL + ks], hb * 64, krow, zk);
                            if (kc >= (uint32_t)C::kStages &&
                                !mbar_wait(&bar[C::VEMPTY + ks], (n - 1) & 1, wctx, 12))
                                goto producer_done;
                            mbar_arrive_expect_tx(&bar[C::VFULL + ks], C::kTile);
#pragma unroll
                            for (int hb = 0; hb < D / 64; ++hb)
                                tma_load_3d(smem + C::kV0 + ks * C::kTile + hb * 16384, &tmv,
                                            &bar[C::VFULL + ks], hb * 64, krow, zk);
                            ++kc;
                        }
                    }
                }
            producer_done:
                // Drain: on an abort, give copies already issued a bounded chance
                // to land before the CTA's shared memory is released.
                if (*abort_flag) {
                    uint64_t t0 = globaltimer_ns();
                    while (globaltimer_ns() - t0 < 2000000ull) {
                    }
                }
            }
        } else if (warp == 8) {
            // ------------------------------------------------------------- MMA issuer
            if (lane == 0) {
                // base descriptors; K steps and stages only advance the start address
                const uint64_t dQ0 = sdesc_sw128(smem_u32(smem + C::kQ0), 16, 1024);
                const uint64_t dK0 = sdesc_sw128(smem_u32(smem + C::kK0), 16, 1024);
                const uint64_t dV0 = sdesc_sw128(smem_u32(smem + C::kV0), 16384, 1024);
                const uint32_t tS0 = tmem, tS1 = tmem + 128;
                const uint32_t tO0 = tmem + 256, tO1 = tmem + 256 + D;
                uint32_t kc = 0, qc = 0, pc0 = 0, pc1 = 0;

                for (int u = blockIdx.x; u < p.total_units; u += gridDim.x) {
                    Unit un = decode_unit(p.units, p.BH, kRowsPerUnit, u, false);
                    const int total = unit_tiles(p, un);
                    if (total == 0)
                        continue;
                    if (!mbar_wait(&bar[C::QFULL], qc & 1, wctx, 20))
                        goto mma_done;
                    ++qc;
                    tc_fence_after();
                    {
                        const int ks = kc % C::kStages;
                        if (!mbar_wait(&bar[C::KFULL + ks], (kc / C::kStages) & 1, wctx, 21))
                            goto mma_done;
                        tc_fence_after();
                        issue_s<D>(tS0, dQ0, dK0, 0, ks * C::kTile);
                        tc_commit(&bar[C::SFULL + 0]);
                        issue_s<D>(tS1, dQ0, dK0, C::kTile, ks * C::kTile);
                        tc_commit(&bar[C::SFULL + 1]);
                        tc_commit(&bar[C::KEMPTY + ks]);
                    }
                    for (int it = 0; it < total; ++it) {
                        const int vs = kc % C::kStages;
                        const bool has_next = it + 1 < total;
                        const int ks2 = (kc + 1) % C::kStages;
                        if (!mbar_wait(&bar[C::VFULL + vs], (kc / C::kStages) & 1, wctx, 22))
                            goto mma_done;
                        if (!mbar_wait(&bar[C::PFULL + 0], pc0 & 1, wctx, 23))
                            goto mma_done;
                        ++pc0;
                        tc_fence_after();
                        issue_pv<D>(tO0, tS0, dV0, vs * C::kTile, it > 0);
                        if (has_next) {
                            if (!mbar_wait(&bar[C::KFULL + ks2], ((kc + 1) / C::kStages) & 1, wctx,
                                           24))
                                goto mma_done;
                            tc_fence_after();
                            issue_s<D>(tS0, dQ0, dK0, 0, ks2 * C::kTile);
                            tc_commit(&bar[C::SFULL + 0]);
                        }
                        if (!mbar_wait(&bar[C::PFULL + 1], pc1 & 1, wctx, 25))
                            goto mma_done;
                        ++pc1;
                        tc_fence_after();
                        issue_pv<D>(tO1, tS1, dV0, vs * C::kTile, it > 0);
                        tc_commit(&bar[C::VEMPTY + vs]);
                        if (has_next) {
                            issue_s<D>(tS1, dQ0, dK0, C::kTile, ks2 * C::kTile);
                            tc_commit(&bar[C::SFULL + 1]);
                            tc_commit(&bar[C::KEMPTY + ks2]);
                        }
                        ++kc;
                    }
                    tc_commit(&bar[C::OFULL + 0]);
                    tc_commit(&bar[C::OFULL + 1]);
                    tc_commit(&bar[C::QEMPTY]);
                }
            mma_done:;
            }
        }
    } else {
        reg_alloc<kRegsMath>();
        // ------------------------------------------------------------- softmax
        const int t = warp >> 2;            // query tile of this warpgroup
        const int wq = warp & 3;            // TMEM lane quarter
        const int rit = wq * 32 + lane;     // row inside the tile
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const uint32_t tS = tmem + lane_off + t * 128;
        const uint32_t tO = tmem + lane_off + 256 + t * D;
        const float c2 = p.scale_log2;
        uint32_t sc = 0, oc = 0;

        for (int u = blockIdx.x; u < p.total_units; u += gridDim.x) {
            Unit un = decode_unit(p.units, p.BH, kRowsPerUnit, u, false);
            const int lrow = un.row0 + t * 128 + rit;
            const bool valid = (t * 128 + rit) < un.nvalid;
            const int32_t pq = valid ? map_pos(p.qmap[un.chunk], lrow) : 0;
            const size_t orow = (size_t)un.slice * p.Lq + (size_t)un.chunk * p.chunk_q + lrow;
            const int total = unit_tiles(p, un);
            float m_ref = -INFINITY, l = 0.f;

            if (total > 0) {
                for (int s = 0; s < p.nkv; ++s) {
                    StepTiles st = step_tiles(p, un, s);
                    if (st.jv <= st.j0)
                        continue;
                    // this row's visible keys of the chunk: rows [lo, cnt)
                    int32_t dlo, dhi;
                    doc_range(p.docs, p.ndocs, pq, dlo, dhi);
                    const int32_t cnt =
                        !valid ? 0 : map_count_le(p.kmap[st.c], p.causal ? pq : dhi - 1);
                    const int32_t lo = map_count_le(p.kmap[st.c], dlo - 1);
                    for (int j = st.j0; j < st.jv; ++j) {
                        if (!mbar_wait(&bar[C::SFULL + t], sc & 1, wctx, 30 + t))
                            goto softmax_done;
                        ++sc;
                        tc_fence_after();
                        uint32_t r[128];
                        tmem_ld32(tS + 0, r);
                        tmem_ld32(tS + 32, r + 32);
                        tmem_ld32(tS + 64, r + 64);
                        tmem_ld32(tS + 96, r + 96);
                        tmem_ld_wait();
                        tmem_reg_fence32(r);
                        tmem_reg_fence32(r + 32);
                        tmem_reg_fence32(r + 64);
                        tmem_reg_fence32(r + 96);
                        float sv[128];
#pragma unroll
                        for (int i = 0; i < 128; ++i)
                            sv[i] = __uint_as_float(r[i]);
                        if (j < st.jf0 || j >= st.jf || !valid) {
                            const int nv = cnt - j * 128, n0 = lo - j * 128;
                            if (n0 <= 0) {
                                // no lower bound inside the tile (always so
                                // without documents): one compare per key
#pragma unroll
                                for (int i = 0; i < 128; ++i)
                                    sv[i] = i < nv ? sv[i] : -INFINITY;
                            } else {
#pragma unroll
                                for (int i = 0; i < 128; ++i)
                                    sv[i] = (i >= n0 && i < nv) ? sv[i] : -INFINITY;
                            }
                        }
                        // row max, two new values per 3-input max
                        float mx = fmaxf(sv[0], sv[1]);
#pragma unroll
                        for (int i = 2; i < 128; i += 2)
                            mx = fmax3(mx, sv[i], sv[i + 1]);
                        const float m_new = fmaxf(m_ref, mx);
                        // Lazy rescale: keep the old reference max unless the
                        // row max grew by more than 2^8 in the exp2 domain.
                        bool grow = m_new > m_ref;
                        bool need = grow && m_ref != -INFINITY && (m_new - m_ref) * c2 > kRescaleLog2;
                        float alpha = 1.f;
                        if (need) {
                            alpha = ex2((m_ref - m_new) * c2);
                            l *= alpha;
                            m_ref = m_new;
                        } else if (grow && m_ref == -INFINITY) {
                            m_ref = m_new;
                        }
                        if (__any_sync(0xffffffffu, need)) {
#pragma unroll 1
                            for (int c0 = 0; c0 < D; c0 += 32) {
                                uint32_t o[32];
                                tmem_ld32(tO + c0, o);
                                tmem_ld_wait();
                                tmem_reg_fence32(o);
#pragma unroll
                                for (int i = 0; i < 32; ++i)
                                    o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                                tmem_st32(tO + c0, o);
                            }
                        }
                        const float mb = (m_ref == -INFINITY) ? 0.f : m_ref * c2;
                        const uint64_t c2x2 = f2pack(c2, c2), nmb2 = f2pack(-mb, -mb);
                        uint32_t pk[64];
                        // two partial sums so that the packed adds are independent
                        uint64_t sum2a = f2pack(0.f, 0.f), sum2b = f2pack(0.f, 0.f);
#pragma unroll
                        for (int i = 0; i < 64; ++i) {
                            float x0, x1;
                            f2unpack(f2fma(f2pack(sv[2 * i], sv[2 * i + 1]), c2x2, nmb2), x0, x1);
                            const float a = ex2(x0), b2 = ex2(x1);
                            if (i & 1)
                                sum2b = f2add(sum2b, f2pack(a, b2));
                            else
                                sum2a = f2add(sum2a, f2pack(a, b2));
                            pk[i] = pack_bf16x2(a, b2);
                        }
                        float s0, s1, s2, s3;
                        f2unpack(sum2a, s0, s1);
                        f2unpack(sum2b, s2, s3);
                        l += (s0 + s1) + (s2 + s3);
                        tmem_st32(tS + 0, pk);
                        tmem_st32(tS + 32, pk + 32);
                        tmem_st_wait();
                        tc_fence_before();
                        mbar_arrive(&bar[C::PFULL + t]);
                    }
                }
                if (!mbar_wait(&bar[C::OFULL + t], oc & 1, wctx, 40 + t))
                    goto softmax_done;
                ++oc;
                tc_fence_after();
            }
            {
                // epilogue: O / l and LSE for valid rows
                const float inv = (l > 0.f) ? 1.f / l : 0.f;
#pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t o[32];
                    if (total > 0) {
                        tmem_ld32(tO + c0, o);
                        tmem_ld_wait();
                        tmem_reg_fence32(o);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            o[i] = 0u;
                    }
                    if (valid && in_bounds(p.status, orow < (size_t)p.BH * p.Lq, 1,
                                           (long long)orow)) {
                        if (p.o_fp32) {
                            float4* dst = reinterpret_cast<float4*>(
                                reinterpret_cast<float*>(p.o) + orow * D + c0);
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                dst[i] = make_float4(__uint_as_float(o[4 * i]) * inv,
                                                     __uint_as_float(o[4 * i + 1]) * inv,
                                                     __uint_as_float(o[4 * i + 2]) * inv,
                                                     __uint_as_float(o[4 * i + 3]) * inv);
                        } else {
                            uint4* dst = reinterpret_cast<uint4*>(
                                reinterpret_cast<__nv_bfloat16*>(p.o) + orow * D + c0);
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                dst[i] = make_uint4(
                                    pack_bf16x2(__uint_as_float(o[8 * i + 0]) * inv,
                                                __uint_as_float(o[8 * i + 1]) * inv),
                                    pack_bf16x2(__uint_as_float(o[8 * i + 2]) * inv,
                                                __uint_as_float(o[8 * i + 3]) * inv),
                                    pack_bf16x2(__uint_as_float(o[8 * i + 4]) * inv,
                                                __uint_as_float(o[8 * i + 5]) * inv),
                                    pack_bf16x2(__uint_as_float(o[8 * i + 6]) * inv,
                                                __uint_as_float(o[8 * i + 7]) * inv));
                        }
                    }
                }
                if (valid && in_bounds(p.status, orow < (size_t)p.BH * p.Lq, 2, (long long)orow))
                    p.lse[orow] = (l > 0.f) ? (m_ref * p.scale + lg2(l) * 0.69314718055994531f)
                                            : -INFINITY;
                tc_fence_before();
            }
        }
    softmax_done:;
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 8) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace fwd

// Host-side launch (declared in dfa_launch.h).
cudaError_t launch_attn_fwd(int d, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const FwdParams& p, int grid,
                            cudaStream_t stream)
{
    if (d == 128) {
        constexpr int smem = fwd::Cfg<128>::kSmem;
        cudaError_t e = cudaFuncSetAttribute(fwd::attn_fwd_kernel<128>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess)
            return e;
        fwd::attn_fwd_kernel<128><<<grid, fwd::kThreads, smem, stream>>>(tq, tk, tv, p);
    } else {
        constexpr int smem = fwd::Cfg<64>::kSmem;
        cudaError_t e = cudaFuncSetAttribute(fwd::attn_fwd_kernel<64>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess)
            return e;
        fwd::attn_fwd_kernel<64><<<grid, fwd::kThreads, smem, stream>>>(tq, tk, tv, p);
    }
    return cudaGetLastError();
}

int fwd_rows_per_unit() { return fwd::kRowsPerUnit; }

}  // namespace dfa
