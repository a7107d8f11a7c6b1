// dfa_bwd.cu -- exact attention backward by recomputation on tcgen05 tensor
// cores (sm_103a).
//
// Method (FlashAttention glossary entry: the softmax is recomputed in the
// backward pass from per-row statistics instead of storing the N x N matrix;
// the gradient formulas are the analytic gradients of exact attention):
//   P = exp(scale Q K^T - LSE),  dV = P^T dO,  dP = dO V^T,
//   dS = P o (dP - D) with D_i = dO_i . O_i,  dQ = scale dS K,
//   dK = scale dS^T Q.
// Masking and tile skipping follow the forward (Striped Attention Guide,
// "Intra-Block vs. Inter-Block Masking Logic").
//
// GB300 mapping (one persistent CTA per SM, 384 threads = 3 warpgroups;
// warps 10-11 only give their registers to the math warpgroups).  A work unit is one
// 128-row key/value tile; it meets every query tile (BQ rows) of every query
// head of its group that can see it.  Everything is computed transposed
// (key rows on TMEM lanes) so that dK and dV stay in TMEM for the whole unit:
//   warp 9      producer: K, V once per unit (TMA); per step the Q and dO
//               tiles (TMA) and the LSE / D values (plain loads) into a
//               2-stage ring.
//   warp 8      MMA issuer: S^T = K Q^T, dP^T = V dO^T (SMEM x SMEM);
//               dV += P^T dO and dK += dS^T Q with P^T / dS^T read from TMEM;
//               dQ from dS^T in SMEM (d = 128: dQ^T = K^T dS^T; d = 64:
//               dQ = dS K).
//   warps 0-3   one thread per key row: P^T, dS^T from S^T, dP^T; writes them
//               to TMEM (bf16) and dS^T to 128-byte-swizzled SMEM; at the end
//               of the unit scales and stores dK, dV.
//   warps 4-7   read the step's dQ tile from TMEM and add it into the fp32
//               dQ accumulator (coalesced atomics).
// TMEM columns: dK [0,d) dV [d,2d) S^T [2d,2d+BQ) dP^T [2d+BQ,2d+2BQ)
// dQ [2d+2BQ, 2d+2BQ+64).
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "dfa_params.h"
#include "dfa_ptx.cuh"

namespace dfa {

namespace bwd {

constexpr int kThreads = 384;      // three warpgroups
// Launch: 384 threads x 168 registers = 64512.  The producer/MMA warpgroup
// drops to 40, the two math warpgroups rise to 232: 128 * (232 + 232 + 40)
// = 64512, the launch's total.
constexpr int kRegsMath = 192;
constexpr int kRegsCtl = 120;
constexpr int kKvRows = 128;

template <int D>
struct Cfg {
    static constexpr int BQ = (D == 128) ? 64 : 128;       // query rows per step
    static constexpr int kKvTile = 128 * D * 2;            // K or V tile bytes
    static constexpr int kQTile = BQ * D * 2;              // Q or dO tile bytes
    static constexpr int kDsBytes = 128 * BQ * 2;          // dS^T tile bytes
    static constexpr int kQStages = 3;                      // Q / dO / LSE / D ring
    static constexpr int kK = 0;
    static constexpr int kV = kK + kKvTile;
    static constexpr int kQ0 = kV + kKvTile;                 // kQStages stages
    static constexpr int kDO0 = kQ0 + kQStages * kQTile;     // kQStages stages
    static constexpr int kDs0 = kDO0 + kQStages * kQTile;    // 2 buffers
    static constexpr int kLse0 = kDs0 + 2 * kDsBytes;        // kQStages x BQ floats
    static constexpr int kDel0 = kLse0 + kQStages * BQ * 4;
    static constexpr int kBar = kDel0 + kQStages * BQ * 4;
    static constexpr int KVFULL = 0, KVEMPTY = 1, QFULL = 2, QEMPTY = QFULL + kQStages,
                         SFULL = QEMPTY + kQStages, PFULL = SFULL + 1, DSFULL = PFULL + 1,
                         DSEMPTY = DSFULL + 1, DQFULL = DSEMPTY + 2, DQEMPTY = DQFULL + 1,
                         DKVFULL = DQEMPTY + 1, NBAR = DKVFULL + 1;
    static constexpr int kSmem = kBar + NBAR * 8 + 16 + 1024;
    // TMEM columns
    static constexpr uint32_t cDK = 0, cDV = D, cS = 2 * D, cDP = 2 * D + BQ,
                              cDQ = 2 * D + 2 * BQ;
};

// Query tiles of chunk p that the unit's key rows can see: [i0, nqt); tiles
// with index >= ifull (and complete) need no mask.
struct QRange {
    int32_t p, i0, nqt, ifull;
};

__device__ __forceinline__ QRange q_range(const BwdParams& pr, const Unit& un, int s, int BQ)
{
    QRange r;
    r.p = pr.ring ? (un.chunk + s) % pr.nq : s;
    r.nqt = ceil_div(pr.chunk_q, BQ);
    if (!pr.causal) {
        r.i0 = 0;
        r.ifull = 0;
        return r;
    }
    const DevMap& km = pr.kmap[un.chunk];
    const DevMap& qm = pr.qmap[r.p];
    const int32_t pk_min = map_pos(km, un.row0);
    const int32_t pk_max = map_pos(km, un.row0 + un.nvalid - 1);
    // first query row whose position is >= pk (positions increase along the chunk)
    const int32_t first_vis = map_count_le(qm, pk_min - 1);
    const int32_t first_full = map_count_le(qm, pk_max - 1);
    r.i0 = first_vis / BQ;
    r.ifull = ceil_div(first_full, BQ);
    if (first_vis >= pr.chunk_q)
        r.i0 = r.nqt;
    return r;
}

__device__ __forceinline__ int32_t unit_steps(const BwdParams& pr, const Unit& un, int BQ)
{
    int32_t t = 0;
    for (int s = 0; s < pr.nq; ++s) {
        QRange r = q_range(pr, un, s, BQ);
        t += r.nqt - r.i0;
    }
    return t * pr.G;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                    const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmdo,
                    const __grid_constant__ BwdParams p)
{
    using C = Cfg<D>;
    constexpr int BQ = C::BQ;
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
        mbar_init(&bar[C::KVFULL], 1);
        mbar_init(&bar[C::KVEMPTY], 1);
        for (int s = 0; s < C::kQStages; ++s) {
            mbar_init(&bar[C::QFULL + s], 1);
            mbar_init(&bar[C::QEMPTY + s], 1);
        }
        mbar_init(&bar[C::SFULL], 1);
        mbar_init(&bar[C::PFULL], 128);
        mbar_init(&bar[C::DSFULL], 128);
        mbar_init(&bar[C::DSEMPTY + 0], 1);
        mbar_init(&bar[C::DSEMPTY + 1], 1);
        mbar_init(&bar[C::DQFULL], 1);
        mbar_init(&bar[C::DQEMPTY], 128);
        mbar_init(&bar[C::DKVFULL], 1);
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
                prefetch_tmap(&tmdo);
            }
            uint32_t uc = 0, qc = 0;
            for (int u = blockIdx.x; u < p.total_units; u += gridDim.x) {
                Unit un = decode_unit(p.units, p.BHkv, kKvRows, u, true);
                if (unit_steps(p, un, BQ) == 0)
                    continue;
                const int b = un.slice / p.Hkv, hk = un.slice % p.Hkv;
                if (lane == 0) {
                    if (uc > 0 && !mbar_wait(&bar[C::KVEMPTY], (uc - 1) & 1, wctx, 50))
                        *abort_flag = 1u;
                    if (!*abort_flag) {
                        mbar_arrive_expect_tx(&bar[C::KVFULL], 2 * C::kKvTile);
                        const int krow = un.chunk * p.chunk_k + un.row0;
#pragma unroll
                        for (int hb = 0; hb < D / 64; ++hb) {
                            tma_load_3d(smem + C::kK + hb * 16384, &tmk, &bar[C::KVFULL], hb * 64, krow,
                                        un.slice);
                            tma_load_3d(smem + C::kV + hb * 16384, &tmv, &bar[C::KVFULL], hb * 64, krow,
                                        un.slice);
                        }
                    }
                }
                __syncwarp();
                if (*abort_flag)
                    goto producer_done;
                ++uc;
                for (int g = 0; g < p.G; ++g) {
                    const int slice_q = b * p.Hq + hk * p.G + g;
                    for (int s = 0; s < p.nq; ++s) {
                        QRange qr = q_range(p, un, s, BQ);
                        for (int i = qr.i0; i < qr.nqt; ++i) {
                            const int st = qc % C::kQStages;
                            const uint32_t use = qc / C::kQStages;
                            if (lane == 0 && use > 0 &&
                                !mbar_wait(&bar[C::QEMPTY + st], (use - 1) & 1, wctx, 51))
                                *abort_flag = 1u;
                            __syncwarp();
                            if (*abort_flag)
                                goto producer_done;
                            // LSE (as log2 units, -inf -> +inf so that P = 0) and D
                            const int32_t m0 = i * BQ;
                            const size_t rbase =
                                (size_t)slice_q * p.Lq + (size_t)qr.p * p.chunk_q + m0;
                            float* sl = (float*)(smem + C::kLse0 + st * BQ * 4);
                            float* sd = (float*)(smem + C::kDel0 + st * BQ * 4);
                            for (int c = lane; c < BQ; c += 32) {
                                float l2 = INFINITY, dl = 0.f;
                                if (m0 + c < p.chunk_q) {
                                    const float lv = p.lse[rbase + c];
                                    l2 = (lv == -INFINITY) ? INFINITY : lv * 1.4426950408889634f;
                                    dl = p.delta[rbase + c];
                                }
                                sl[c] = l2;
                                sd[c] = dl;
                            }
                            __syncwarp();
                            if (lane == 0) {
                                mbar_arrive_expect_tx(&bar[C::QFULL + st], 2 * C::kQTile);
                                const int qrow = qr.p * p.chunk_q + m0;
#pragma unroll
                                for (int hb = 0; hb < D / 64; ++hb) {
                                    tma_load_3d(smem + C::kQ0 + st * C::kQTile + hb * (BQ * 128), &tmq,
                                                &bar[C::QFULL + st], hb * 64, qrow, slice_q);
                                    tma_load_3d(smem + C::kDO0 + st * C::kQTile + hb * (BQ * 128),
                                                &tmdo, &bar[C::QFULL + st], hb * 64, qrow, slice_q);
                                }
                            }
                            ++qc;
                        }
                    }
                }
            }
        producer_done:
            if (lane == 0 && *abort_flag) {
                uint64_t t0 = globaltimer_ns();
                while (globaltimer_ns() - t0 < 2000000ull) {
                }
            }
        } else if (warp == 8) {
            // ------------------------------------------------------------- MMA issuer
            if (lane == 0) {
                constexpr uint32_t idSt = idesc_bf16_f32(128, BQ, false, false);
                constexpr uint32_t idKV = idesc_bf16_f32(128, D, false, true);
                constexpr uint32_t idQ = idesc_bf16_f32(128, 64, true, true);
                const uint32_t sK = smem_u32(smem + C::kK), sV = smem_u32(smem + C::kV);
                const uint32_t sQ = smem_u32(smem + C::kQ0), sDO = smem_u32(smem + C::kDO0);
                const uint32_t sDs0 = smem_u32(smem + C::kDs0);
                uint32_t uc = 0, n = 0;

                // S^T = K Q^T and dP^T = V dO^T for stage st
                auto issue_sdp = [&](int st) {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t ka = (kk >> 2) * 16384 + (kk & 3) * 32;
                        const uint32_t qa = st * C::kQTile + (kk >> 2) * (BQ * 128) + (kk & 3) * 32;
                        mma_ss(tmem + C::cS, sdesc_sw128(sK + ka, 16, 1024),
                               sdesc_sw128(sQ + qa, 16, 1024), idSt, kk > 0);
                        mma_ss(tmem + C::cDP, sdesc_sw128(sV + ka, 16, 1024),
                               sdesc_sw128(sDO + qa, 16, 1024), idSt, kk > 0);
                    }
                };

                for (int u = blockIdx.x; u < p.total_units; u += gridDim.x) {
                    Unit un = decode_unit(p.units, p.BHkv, kKvRows, u, true);
                    const int T = unit_steps(p, un, BQ);
                    if (T == 0)
                        continue;
                    if (!mbar_wait(&bar[C::KVFULL], uc & 1, wctx, 60))
                        goto mma_done;
                    ++uc;
                    tc_fence_after();
                    if (!mbar_wait(&bar[C::QFULL + n % C::kQStages], (n / C::kQStages) & 1, wctx,
                                   61))
                        goto mma_done;
                    tc_fence_after();
                    issue_sdp(n % C::kQStages);
                    tc_commit(&bar[C::SFULL]);
                    for (int it = 0; it < T; ++it, ++n) {
                        const int st = n % C::kQStages;
                        if (!mbar_wait(&bar[C::PFULL], n & 1, wctx, 62))
                            goto mma_done;
                        tc_fence_after();
                        // dV += P^T dO
#pragma unroll
                        for (int kk = 0; kk < BQ / 16; ++kk)
                            mma_ts(tmem + C::cDV, tmem + C::cS + kk * 8,
                                   sdesc_sw128(sDO + st * C::kQTile + kk * 2048, BQ * 128, 1024), idKV,
                                   (it > 0 || kk > 0) ? 1u : 0u);
                        if (!mbar_wait(&bar[C::DSFULL], n & 1, wctx, 63))
                            goto mma_done;
                        tc_fence_after();
                        // dK += dS^T Q
#pragma unroll
                        for (int kk = 0; kk < BQ / 16; ++kk)
                            mma_ts(tmem + C::cDK, tmem + C::cDP + kk * 8,
                                   sdesc_sw128(sQ + st * C::kQTile + kk * 2048, BQ * 128, 1024), idKV,
                                   (it > 0 || kk > 0) ? 1u : 0u);
                        tc_commit(&bar[C::QEMPTY + st]);
                        if (it + 1 < T) {
                            const uint32_t n2 = n + 1;
                            if (!mbar_wait(&bar[C::QFULL + n2 % C::kQStages],
                                           (n2 / C::kQStages) & 1, wctx, 64))
                                goto mma_done;
                            tc_fence_after();
                            issue_sdp(n2 % C::kQStages);
                            tc_commit(&bar[C::SFULL]);
                        }
                        if (n > 0 && !mbar_wait(&bar[C::DQEMPTY], (n - 1) & 1, wctx, 65))
                            goto mma_done;
                        tc_fence_after();
                        // dQ for this step from dS^T in shared memory (buffer n & 1)
                        const uint32_t sDs = sDs0 + (n & 1) * C::kDsBytes;
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) {
                            if (D == 128) {
                                // dQ^T [d x BQ] = K^T [d x kv] dS^T [kv x BQ]
                                mma_ss(tmem + C::cDQ, sdesc_sw128(sK + kk * 2048, 16384, 1024),
                                       sdesc_sw128(sDs + kk * 2048, 16384, 1024), idQ, kk > 0);
                            } else {
                                // dQ [BQ x d] = dS [BQ x kv] K [kv x d]
                                mma_ss(tmem + C::cDQ, sdesc_sw128(sDs + kk * 2048, 16384, 1024),
                                       sdesc_sw128(sK + kk * 2048, 16384, 1024), idQ, kk > 0);
                            }
                        }
                        tc_commit(&bar[C::DQFULL]);
                        tc_commit(&bar[C::DSEMPTY + (n & 1)]);
                    }
                    tc_commit(&bar[C::DKVFULL]);
                    tc_commit(&bar[C::KVEMPTY]);
                }
            mma_done:;
            }
        }
    } else if (warp < 4) {
        // ------------------------------------------------------------- P^T, dS^T
        reg_alloc<kRegsMath>();
        const int r = warp * 32 + lane;  // key row inside the unit tile (TMEM lane)
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        const float c2 = p.scale_log2;
        uint32_t n = 0, uc = 0;
        for (int u = blockIdx.x; u < p.total_units; u += gridDim.x) {
            Unit un = decode_unit(p.units, p.BHkv, kKvRows, u, true);
            const int T = unit_steps(p, un, BQ);
            const bool kvalid = r < un.nvalid;
            const int32_t pk = kvalid ? map_pos(p.kmap[un.chunk], un.row0 + r) : 0;
            if (T > 0) {
                for (int g = 0; g < p.G; ++g) {
                    for (int s = 0; s < p.nq; ++s) {
                        QRange qr = q_range(p, un, s, BQ);
                        if (qr.i0 >= qr.nqt)
                            continue;
                        // first query row of chunk qr.p that sees this key row
                        const int32_t qv =
                            !kvalid ? 0x7fffffff
                                    : (p.causal ? map_count_le(p.qmap[qr.p], pk - 1) : 0);
                        for (int i = qr.i0; i < qr.nqt; ++i, ++n) {
                            const int st = n % C::kQStages;
                            if (!mbar_wait(&bar[C::QFULL + st], (n / C::kQStages) & 1, wctx, 70))
                                goto sm_done;
                            if (!mbar_wait(&bar[C::SFULL], n & 1, wctx, 71))
                                goto sm_done;
                            // the dQ MMA of two steps ago has read this dS^T buffer
                            if (n >= 2 &&
                                !mbar_wait(&bar[C::DSEMPTY + (n & 1)], ((n >> 1) - 1) & 1, wctx, 72))
                                goto sm_done;
                            tc_fence_after();
                            const float* sl = (const float*)(smem + C::kLse0 + st * BQ * 4);
                            const float* sd = (const float*)(smem + C::kDel0 + st * BQ * 4);
                            const bool full = (i >= qr.ifull) && ((i + 1) * BQ <= p.chunk_q) &&
                                              un.nvalid == kKvRows;
                            // 32 query columns at a time: P^T = exp2(S^T c - LSE log2e),
                            // dS^T = P^T (dP^T - D); bf16 P^T over S^T and dS^T over dP^T
                            // in TMEM, dS^T also to the swizzled SMEM tile.
#pragma unroll 1
                            for (int c0 = 0; c0 < BQ; c0 += 32) {
                                uint32_t sr[32], dr[32];
                                tmem_ld32(tmem + lane_off + C::cS + c0, sr);
                                tmem_ld32(tmem + lane_off + C::cDP + c0, dr);
                                tmem_ld_wait();
                                tmem_reg_fence32(sr);
                                tmem_reg_fence32(dr);
                                uint32_t pp[16], dd[16];
#pragma unroll
                                for (int c4 = 0; c4 < 8; ++c4) {
                                    const float4 l4 = *(const float4*)(sl + c0 + 4 * c4);
                                    const float4 d4 = *(const float4*)(sd + c0 + 4 * c4);
                                    const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
                                    const float dv[4] = {d4.x, d4.y, d4.z, d4.w};
                                    float pv[4], ds[4];
#pragma unroll
                                    for (int e = 0; e < 4; ++e) {
                                        const int c = 4 * c4 + e;
                                        float pe = ex2(fmaf(__uint_as_float(sr[c]), c2, -lv[e]));
                                        if (!full) {
                                            const int q = i * BQ + c0 + c;
                                            pe = (q >= qv && q < p.chunk_q) ? pe : 0.f;
                                        }
                                        pv[e] = pe;
                                        ds[e] = pe * (__uint_as_float(dr[c]) - dv[e]);
                                    }
                                    pp[2 * c4] = pack_bf16x2(pv[0], pv[1]);
                                    pp[2 * c4 + 1] = pack_bf16x2(pv[2], pv[3]);
                                    dd[2 * c4] = pack_bf16x2(ds[0], ds[1]);
                                    dd[2 * c4 + 1] = pack_bf16x2(ds[2], ds[3]);
                                }
                                tmem_st16(tmem + lane_off + C::cS + c0 / 2, pp);
                                tmem_st16(tmem + lane_off + C::cDP + c0 / 2, dd);
                                // 32 bf16 = four 16-byte chunks of row r in block c0 / 64
                                uint8_t* blk =
                                    smem + C::kDs0 + (n & 1) * C::kDsBytes + (c0 / 64) * 16384;
#pragma unroll
                                for (int ch = 0; ch < 4; ++ch)
                                    *(uint4*)(blk + sw128_offset(r, (c0 % 64) / 8 + ch)) =
                                        make_uint4(dd[4 * ch], dd[4 * ch + 1], dd[4 * ch + 2],
                                                   dd[4 * ch + 3]);
                            }
                            tmem_st_wait();
                            fence_proxy_async_smem();
                            tc_fence_before();
                            mbar_arrive(&bar[C::PFULL]);
                            mbar_arrive(&bar[C::DSFULL]);
                        }
                    }
                }
                if (!mbar_wait(&bar[C::DKVFULL], uc & 1, wctx, 73))
                    goto sm_done;
                ++uc;
                tc_fence_after();
            }
            {
                // epilogue: dK (scaled) and dV rows of the unit
                const size_t orow =
                    (size_t)un.slice * p.Lk + (size_t)un.chunk * p.chunk_k + un.row0 + r;
#pragma unroll 1
                for (int which = 0; which < 2; ++which) {
                    const uint32_t col = which == 0 ? C::cDK : C::cDV;
                    const float mul = which == 0 ? p.scale : 1.f;
                    void* outp = which == 0 ? p.dk : p.dv;
#pragma unroll 1
                    for (int c0 = 0; c0 < D; c0 += 32) {
                        uint32_t o[32];
                        if (T > 0) {
                            tmem_ld32(tmem + lane_off + col + c0, o);
                            tmem_ld_wait();
                            tmem_reg_fence32(o);
                        } else {
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                o[e] = 0u;
                        }
                        if (!kvalid)
                            continue;
                        if (p.dkv_mode == 0) {
                            uint4* dst = reinterpret_cast<uint4*>(
                                reinterpret_cast<__nv_bfloat16*>(outp) + orow * D + c0);
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                dst[e] = make_uint4(
                                    pack_bf16x2(__uint_as_float(o[8 * e + 0]) * mul,
                                                __uint_as_float(o[8 * e + 1]) * mul),
                                    pack_bf16x2(__uint_as_float(o[8 * e + 2]) * mul,
                                                __uint_as_float(o[8 * e + 3]) * mul),
                                    pack_bf16x2(__uint_as_float(o[8 * e + 4]) * mul,
                                                __uint_as_float(o[8 * e + 5]) * mul),
                                    pack_bf16x2(__uint_as_float(o[8 * e + 6]) * mul,
                                                __uint_as_float(o[8 * e + 7]) * mul));
                        } else {
                            float4* dst = reinterpret_cast<float4*>(
                                reinterpret_cast<float*>(outp) + orow * D + c0);
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                float4 a = dst[e];
                                a.x += __uint_as_float(o[4 * e + 0]) * mul;
                                a.y += __uint_as_float(o[4 * e + 1]) * mul;
                                a.z += __uint_as_float(o[4 * e + 2]) * mul;
                                a.w += __uint_as_float(o[4 * e + 3]) * mul;
                                dst[e] = a;
                            }
                        }
                    }
                }
                tc_fence_before();
            }
        }
    sm_done:;
    } else {
        // ------------------------------------------------------------- dQ drain
        reg_alloc<kRegsMath>();
        const int wq = warp & 3;
        const int L = wq * 32 + lane;  // TMEM lane of this thread
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        uint32_t n = 0;
        for (int u = blockIdx.x; u < p.total_units; u += gridDim.x) {
            Unit un = decode_unit(p.units, p.BHkv, kKvRows, u, true);
            if (unit_steps(p, un, BQ) == 0)
                continue;
            const int b = un.slice / p.Hkv, hk = un.slice % p.Hkv;
            for (int g = 0; g < p.G; ++g) {
                const int slice_q = b * p.Hq + hk * p.G + g;
                for (int s = 0; s < p.nq; ++s) {
                    QRange qr = q_range(p, un, s, BQ);
                    for (int i = qr.i0; i < qr.nqt; ++i, ++n) {
                        if (!mbar_wait(&bar[C::DQFULL], n & 1, wctx, 80))
                            goto dq_done;
                        tc_fence_after();
                        uint32_t v[64];
                        tmem_ld32(tmem + lane_off + C::cDQ, v);
                        tmem_ld32(tmem + lane_off + C::cDQ + 32, v + 32);
                        tmem_ld_wait();
                        tmem_reg_fence32(v);
                        tmem_reg_fence32(v + 32);
                        tc_fence_before();
                        mbar_arrive(&bar[C::DQEMPTY]);
                        const int m0 = i * BQ;
                        float* base = p.dq_acc +
                                      ((size_t)slice_q * p.Lq + (size_t)qr.p * p.chunk_q) * D;
                        if (D == 128) {
                            // lane = feature column, columns = query rows m0 .. m0+63
#pragma unroll
                            for (int c = 0; c < 64; ++c)
                                if (m0 + c < p.chunk_q)
                                    atomicAdd(base + (size_t)(m0 + c) * D + L,
                                              __uint_as_float(v[c]) * p.scale);
                        } else {
                            // lane = query row, columns = features
                            if (m0 + L < p.chunk_q) {
                                float4* dst =
                                    reinterpret_cast<float4*>(base + (size_t)(m0 + L) * D);
#pragma unroll
                                for (int e = 0; e < 16; ++e)
                                    atomicAdd(dst + e,
                                              make_float4(__uint_as_float(v[4 * e]) * p.scale,
                                                          __uint_as_float(v[4 * e + 1]) * p.scale,
                                                          __uint_as_float(v[4 * e + 2]) * p.scale,
                                                          __uint_as_float(v[4 * e + 3]) * p.scale));
                            }
                        }
                    }
                }
            }
        }
    dq_done:;
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 8) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace bwd

cudaError_t launch_attn_bwd(int d, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& tdo, const BwdParams& p,
                            int grid, cudaStream_t stream)
{
    if (d == 128) {
        constexpr int smem = bwd::Cfg<128>::kSmem;
        cudaError_t e = cudaFuncSetAttribute(bwd::attn_bwd_kernel<128>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess)
            return e;
        bwd::attn_bwd_kernel<128><<<grid, bwd::kThreads, smem, stream>>>(tq, tk, tv, tdo, p);
    } else {
        constexpr int smem = bwd::Cfg<64>::kSmem;
        cudaError_t e = cudaFuncSetAttribute(bwd::attn_bwd_kernel<64>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess)
            return e;
        bwd::attn_bwd_kernel<64><<<grid, bwd::kThreads, smem, stream>>>(tq, tk, tv, tdo, p);
    }
    return cudaGetLastError();
}

int bwd_rows_per_unit() { return bwd::kKvRows; }

}  // namespace dfa
