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
// GB300 mapping: one persistent CTA per SM, 512 threads = 4 warpgroups.  A
// work unit is one 128-row key/value tile; it meets every visible 128-row
// query tile ("step") of every query head of its group, the group's query
// heads innermost (all of them at one query tile before the next tile), so
// that the units running at one time work on the same query rows of every
// head of the group.  Key rows sit on TMEM
// lanes, so dK and dV accumulate in TMEM for the whole unit.  Every product
// of a step is an M = 128, N = 128 (or N = d) tcgen05 MMA: the K, V and K^T
// operands are read from shared memory once per 128 query rows, and no
// instruction asks shared memory for more bytes per cycle than it delivers.
//   warp 13     producer: K, V once per unit (TMA); per step the Q tile with
//               its rows' -LSE/scale records into a 2-stage ring, and the dO
//               tile with its rows' -D records into a single stage that is
//               refilled as soon as dP^T and dV of the step have read it.
//   warp 14     issues S^T = K Q^T - LSE/scale (once dK of the previous step
//               has read the dS^T packed into the S^T columns; dV, issued
//               before dK, has read P^T there) and
//               dP^T = V dO^T - D (once the previous dQ^T has been drained
//               from the columns dP^T overwrites).  The row constants enter
//               as one more K = 16 slice of each product: a ones tile against
//               per-row records holding the constant split into three bf16
//               values (hi + mid + lo, exact to fp32 precision), so the
//               softmax warps read no per-row data.  S^T and dP^T signal
//               completion separately.
//   warp 12     issues dV += P^T dO (on P^T ready), then, on dS^T ready,
//               dQ^T = K^T dS^T into the dP^T columns (B operand: the dS^T
//               tile in shared memory) and dK += dS^T Q (A operand: dS^T
//               packed in TMEM, in the half of the S^T columns that P^T
//               leaves free).  dQ^T goes first: the next dP^T waits for its
//               columns, which the drain frees while dK still runs (dK first
//               cost 4 % at 128K).
//   warps 0-7   two warpgroups, one thread per key row, warpgroup h on query
//               columns [64 h, 64 h + 64) of each step, in two halves of 32:
//               P^T = exp2(S^T c), packed (bf16) into its own columns of the
//               S^T region and signalled; then dS^T = P^T (dP^T - D) packed
//               into the other half of those columns (dK's A operand) and
//               stored into the swizzled SMEM tile that is the B operand of
//               dQ^T.  At the end of a unit the
//               first warpgroup stores dK (scaled), the second dV.
//   warps 8-11  drain each step's dQ^T tile from TMEM (all 128 columns into
//               registers, which frees the columns for the next dP^T) and add
//               it into the fp32 dQ accumulator with coalesced atomics.
//   warp 15     gives its registers to the other warpgroups.
// TMEM columns: dK [0,d) dV [d,2d), S^T [2d, 2d+128), dP^T (later dQ^T)
// [2d+128, 2d+256).  d = 64 uses the same path: the K tile is padded to 128
// columns with zeros so that dQ^T has 128 lanes.
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "dfa_params.h"
#include "dfa_ptx.cuh"

namespace dfa {

namespace bwd {

constexpr int kThreads = 512;
// Launch: 512 threads x 128 registers = 65536.  Rebalanced per warpgroup:
// 128 * (kRegsSoft * 2 + kRegsDrain + kRegsCtl) = 65536.  The drain holds a
// whole dQ^T row (128 values) in registers.
constexpr int kRegsSoft = 128;
constexpr int kRegsDrain = 160;
constexpr int kRegsCtl = 96;
static_assert(2 * kRegsSoft + kRegsDrain + kRegsCtl == 512, "register budget");
constexpr int kWarpMma = 12, kWarpProducer = 13, kWarpMmaS = 14;
constexpr int kKvRows = 128;
constexpr int BQ = 128;  // query rows per step

template <int D>
struct Cfg {
    static constexpr int kKTile = 128 * 128 * 2;  // K tile, always 128 columns (zero padded)
    static constexpr int kVTile = 128 * D * 2;
    static constexpr int kQTile = BQ * D * 2;     // Q or dO tile
    static constexpr int kDsBytes = 128 * BQ * 2; // the dS^T tile (two 64-column blocks)
    static constexpr int kQStages = 2;
    // K = 16 slices that add -LSE/scale to S^T and -D to dP^T: a 128-row
    // ones tile (the key side) and per stage one 128-row record tile (the
    // query side), rows of 32 bytes, 32-byte swizzle
    static constexpr int kAugTile = BQ * 32;
    static constexpr int kK = 0;
    static constexpr int kV = kK + kKTile;
    static constexpr int kQ0 = kV + kVTile;
    static constexpr int kDO = kQ0 + kQStages * kQTile;
    static constexpr int kDs = kDO + kQTile;
    static constexpr int kOnes = kDs + kDsBytes;
    static constexpr int kQA0 = kOnes + 128 * 32;
    static constexpr int kDA = kQA0 + kQStages * kAugTile;
    static constexpr int kBar = kDA + kAugTile;
    // KVFULL/KVEMPTY: the unit's K, V; QFULL/QEMPTY: a Q stage (with its
    // -LSE/scale records); DOFULL/DOEMPTY: the dO stage (with its -D
    // records; emptied by two arrivals: dP^T and dV have read it).
    // SFULL: S^T of a step computed; DPFULL: its dP^T computed; PREADY: its
    // P^T written to TMEM; DSREADY: its dS^T written (TMEM and the SMEM
    // tile); DQFULL: its dQ^T computed; DQEMPTY: dQ^T read out of TMEM (the
    // dP^T columns free); DKDONE: its dK computed (dK is the step's last MMA:
    // the S^T columns, the dS^T tile and the Q stage are all read);
    // DKVFULL: all of the unit's MMAs complete.
    static constexpr int KVFULL = 0, KVEMPTY = 1, QFULL = 2, QEMPTY = QFULL + kQStages,
                         DOFULL = QEMPTY + kQStages, DOEMPTY = DOFULL + 1, SFULL = DOEMPTY + 1,
                         DPFULL = SFULL + 1, PREADY = DPFULL + 1, DSREADY = PREADY + 1,
                         DQFULL = DSREADY + 1, DQEMPTY = DQFULL + 1,
                         DKVFULL = DQEMPTY + 1, DKDONE = DKVFULL + 1, NBAR = DKDONE + 1;
    static constexpr int kSmem = kBar + NBAR * 8 + 16 + 1024;
    static constexpr uint32_t cDK = 0, cDV = D, cS = 2 * D, cDP = 2 * D + 128;
};
static_assert(Cfg<128>::kSmem <= 232448, "shared memory budget");
// Query tiles of chunk p that the unit's key rows can see: [i0, i1); tiles in
// [if0, if1) see every key row (no mask).  A key at position y is seen by the
// queries at positions [causal ? y : doc_lo(y), doc_hi(y) - 1] (its document;
// everything without documents), an interval of each query chunk.  Union over
// the unit's keys: [lower(y_min), doc_hi(y_max) - 1]; intersection:
// [lower(y_max), doc_hi(y_min) - 1], and only when all keys share a document.
struct QRange {
    int32_t p, i0, i1, if0, if1;
};

// Query blocking: a unit covers only the query tiles of its block (the same
// local tile range of every query chunk), so that the units running at one
// time share a bounded set of Q / dO / dQ rows in L2.
__device__ __forceinline__ QRange clamp_block(const BwdParams& pr, const Unit& un, QRange r)
{
    if (pr.nqblk > 1) {
        const int32_t b0 = un.qblk * pr.qblk_tiles, b1 = b0 + pr.qblk_tiles;
        r.i0 = max(r.i0, b0);
        r.i1 = min(r.i1, b1);
    }
    if (r.i1 < r.i0)
        r.i1 = r.i0;
    return r;
}

// Step s visits query chunk s: every unit takes the chunks in the same order
// (not rotated by its own chunk as a ring of workers would), so the units
// running at one time read the same chunk's Q / dO tiles and add into the
// same chunk's dQ rows, out of L2.
__device__ __forceinline__ QRange q_range(const BwdParams& pr, const Unit& un, int s)
{
    QRange r;
    r.p = s;
    const int32_t nqt = ceil_div(pr.chunk_q, BQ);
    if (!pr.causal && pr.ndocs == 0) {
        r.i0 = 0;
        r.i1 = nqt;
        r.if0 = 0;
        r.if1 = pr.chunk_q / BQ;
        return clamp_block(pr, un, r);
    }
    const DevMap& km = pr.kmap[un.chunk];
    const DevMap& qm = pr.qmap[r.p];
    const int32_t pk_min = map_pos(km, un.row0);
    const int32_t pk_max = map_pos(km, un.row0 + un.nvalid - 1);
    int32_t lo_min, hi_min, lo_max, hi_max;
    doc_range(pr.docs, pr.ndocs, pk_min, lo_min, hi_min);
    doc_range(pr.docs, pr.ndocs, pk_max, lo_max, hi_max);
    const int32_t first_vis = map_count_le(qm, (pr.causal ? pk_min : lo_min) - 1);
    const int32_t end_vis = map_count_le(qm, hi_max - 1);
    const int32_t first_full = map_count_le(qm, (pr.causal ? pk_max : lo_max) - 1);
    const int32_t end_full = lo_max <= pk_min ? map_count_le(qm, hi_min - 1) : 0;
    r.i0 = first_vis / BQ;
    r.i1 = ceil_div(end_vis, BQ);
    r.if0 = ceil_div(first_full, BQ);
    r.if1 = end_full / BQ;
    return clamp_block(pr, un, r);
}

// Unit u: slices (b, kv head) outermost, then query blocks, then the key
// units of the slice in the table's order.
__device__ __forceinline__ Unit bwd_unit(const BwdParams& p, int u)
{
    const int ups = p.units.units_per_slice;
    const int per = p.nqblk * ups;
    const int slice = u / per, r = u - slice * per;
    Unit un = decode_unit(p.units, p.BHkv, kKvRows, slice * ups + r % ups, true);
    un.qblk = r / ups;
    return un;
}

__device__ __forceinline__ int32_t unit_steps(const BwdParams& pr, const Unit& un)
{
    int32_t t = 0;
    for (int s = 0; s < pr.nq; ++s) {
        QRange r = q_range(pr, un, s);
        t += r.i1 - r.i0;
    }
    return t * pr.G;
}

// TMEM column of the packed bf16 P^T for K step kk (16 query rows; the
// packed dS^T sits 32 columns further):
// warpgroup h's query columns [64 h, 64 h + 64) are packed at columns
// [64 h, 64 h + 32) of the region (its own columns, so that neither
// warpgroup overwrites values the other has still to read).
__host__ __device__ constexpr uint32_t ptcol(int kk) { return (kk >> 2) * 64 + (kk & 3) * 8; }

struct Shared {
    uint8_t* smem;
    uint64_t* bar;
    volatile uint32_t* abort_flag;
    uint32_t tmem;
};

// ---------------------------------------------------------------------------
// producer (warp 13; lane 0 issues every TMA load: K, V per unit; per step Q
// with its -LSE/scale records, then dO with its -D records)
// ---------------------------------------------------------------------------
template <int D>
__device__ __forceinline__ void producer(const BwdParams& p, const Shared& sh, const WaitCtx& w,
                                         const CUtensorMap* tmq, const CUtensorMap* tmk,
                                         const CUtensorMap* tmv, const CUtensorMap* tmdo,
                                         const CUtensorMap* tmal, const CUtensorMap* tmad)
{
    using C = Cfg<D>;
    const int lane = threadIdx.x & 31;
    uint64_t* bar = sh.bar;
    uint8_t* smem = sh.smem;
    if (lane == 0) {
        prefetch_tmap(tmq);
        prefetch_tmap(tmk);
        prefetch_tmap(tmv);
        prefetch_tmap(tmdo);
        prefetch_tmap(tmal);
        prefetch_tmap(tmad);
    }
    uint32_t uc = 0, qc = 0;
    for (int u = blockIdx.x; u < p.total_units; u += gridDim.x) {
        Unit un = bwd_unit(p, u);
        if (unit_steps(p, un) == 0)
            continue;
        const int b = un.slice / p.Hkv, hk = un.slice % p.Hkv;
        if (lane == 0) {
            if (uc > 0 && !mbar_wait(&bar[C::KVEMPTY], (uc - 1) & 1, w, 50))
                *sh.abort_flag = 1u;
            if (!*sh.abort_flag) {
                mbar_arrive_expect_tx(&bar[C::KVFULL], (D / 64) * 2 * 16384);
                const int krow = un.chunk * p.chunk_k + un.row0;
#pragma unroll
                for (int hb = 0; hb < D / 64; ++hb) {
                    tma_load_3d(smem + C::kK + hb * 16384, tmk, &bar[C::KVFULL], hb * 64, krow,
                                un.slice);
                    tma_load_3d(smem + C::kV + hb * 16384, tmv, &bar[C::KVFULL], hb * 64, krow,
                                un.slice);
                }
            }
        }
        __syncwarp();
        if (*sh.abort_flag)
            return;
        ++uc;
        for (int s = 0; s < p.nq; ++s) {
            QRange qr = q_range(p, un, s);
            for (int i = qr.i0; i < qr.i1; ++i) {
                for (int g = 0; g < p.G; ++g, ++qc) {
                    const int slice_q = b * p.Hq + hk * p.G + g;
                    const int st = qc % C::kQStages;
                    const uint32_t use = qc / C::kQStages;
                    const int qrow = qr.p * p.chunk_q + i * BQ;
                    // rows past the chunk read as the next chunk's (or zeros past
                    // the tensor); their P is masked
                    if (lane == 0) {
                        if (use > 0 && !mbar_wait(&bar[C::QEMPTY + st], (use - 1) & 1, w, 51))
                            *sh.abort_flag = 1u;
                        if (!*sh.abort_flag) {
                            mbar_arrive_expect_tx(&bar[C::QFULL + st], C::kQTile + C::kAugTile);
                            tma_load_3d(smem + C::kQA0 + st * C::kAugTile, tmal,
                                        &bar[C::QFULL + st], 0, qrow, slice_q);
#pragma unroll
                            for (int hb = 0; hb < D / 64; ++hb)
                                tma_load_3d(smem + C::kQ0 + st * C::kQTile + hb * (BQ * 128), tmq,
                                            &bar[C::QFULL + st], hb * 64, qrow, slice_q);
                        }
                        if (!*sh.abort_flag && qc > 0 &&
                            !mbar_wait(&bar[C::DOEMPTY], (qc - 1) & 1, w, 52))
                            *sh.abort_flag = 1u;
                        if (!*sh.abort_flag) {
                            mbar_arrive_expect_tx(&bar[C::DOFULL], C::kQTile + C::kAugTile);
                            tma_load_3d(smem + C::kDA, tmad, &bar[C::DOFULL], 0, qrow, slice_q);
#pragma unroll
                            for (int hb = 0; hb < D / 64; ++hb)
                                tma_load_3d(smem + C::kDO + hb * (BQ * 128), tmdo, &bar[C::DOFULL],
                                            hb * 64, qrow, slice_q);
                        }
                    }
                    __syncwarp();
                    if (*sh.abort_flag)
                        return;
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// MMA issuers (lane 0 of warps 14 and 12)
// ---------------------------------------------------------------------------
// Two threads issue the MMAs, so that one thread's barrier waits are covered
// by the other's issues.  Every dependency between them goes through a
// completion barrier, never through issue order.
//
// Warp 14 (issue_products), per step m:
//   S^T(m) = K Q(m)^T - LSE/scale   once Q(m) has landed and dK(m-1) has
//                                   read dS^T(m-1) from the same columns
//                                   (dV(m-1), issued before it, P^T(m-1));
//   dP^T(m) = V dO(m)^T - D         once dO(m) has landed and dQ^T(m-1) has
//                                   been read out of the same columns.
// Warp 12 (issue_grads), per step n:
//   dV += P^T(n) dO(n)    once the softmax warps have written P^T (and dO(n)
//                         has landed);
//   dQ^T(n) = K^T dS^T(n) into the dP^T columns, once they have written
//                         dS^T (B operand: the SMEM tile);
//   dK += dS^T(n) Q(n)    A operand: dS^T packed in the S^T columns; after
//                         dQ^T so that the drain reads dQ^T (and frees the
//                         dP^T columns) meanwhile.
template <int D>
__device__ __forceinline__ void issue_products(const BwdParams& p, const Shared& sh,
                                               const WaitCtx& w)
{
    using C = Cfg<D>;
    uint64_t* bar = sh.bar;
    const uint32_t tmem = sh.tmem;
    constexpr uint32_t idSt = idesc_bf16_f32(128, BQ, false, false);
    const uint64_t dKk = sdesc_sw128(smem_u32(sh.smem + C::kK), 16, 1024);
    const uint64_t dVk = sdesc_sw128(smem_u32(sh.smem + C::kV), 16, 1024);
    const uint64_t dQk = sdesc_sw128(smem_u32(sh.smem + C::kQ0), 16, 1024);
    const uint64_t dDOk = sdesc_sw128(smem_u32(sh.smem + C::kDO), 16, 1024);
    const uint64_t dOnes = sdesc_sw32(smem_u32(sh.smem + C::kOnes), 256);
    const uint64_t dQA = sdesc_sw32(smem_u32(sh.smem + C::kQA0), 256);
    const uint64_t dDA = sdesc_sw32(smem_u32(sh.smem + C::kDA), 256);
    uint32_t uc = 0, m = 0;
    for (int u = blockIdx.x; u < p.total_units; u += gridDim.x) {
        Unit un = bwd_unit(p, u);
        const int T = unit_steps(p, un);
        if (T == 0)
            continue;
        if (!mbar_wait(&bar[C::KVFULL], uc & 1, w, 60))
            return;
        ++uc;
        for (int it = 0; it < T; ++it, ++m) {
            const uint32_t qs = m % C::kQStages;
            if (!mbar_wait(&bar[C::QFULL + qs], (m / C::kQStages) & 1, w, 61))
                return;
            if (m >= 1 && !mbar_wait(&bar[C::DKDONE], (m - 1) & 1, w, 62))
                return;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
                mma_ss(tmem + C::cS, sdesc_add(dKk, (kk >> 2) * 16384 + (kk & 3) * 32),
                       sdesc_add(dQk, qs * C::kQTile + (kk >> 2) * (BQ * 128) + (kk & 3) * 32),
                       idSt, kk > 0);
            // S^T - LSE/scale: one more K = 16 slice, ones against the records
            mma_ss(tmem + C::cS, dOnes, sdesc_add(dQA, qs * C::kAugTile), idSt, 1u);
            tc_commit(&bar[C::SFULL]);
            if (!mbar_wait(&bar[C::DOFULL], m & 1, w, 64))
                return;
            if (m >= 1 && !mbar_wait(&bar[C::DQEMPTY], (m - 1) & 1, w, 65))
                return;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
                mma_ss(tmem + C::cDP, sdesc_add(dVk, (kk >> 2) * 16384 + (kk & 3) * 32),
                       sdesc_add(dDOk, (kk >> 2) * (BQ * 128) + (kk & 3) * 32), idSt, kk > 0);
            // dP^T - D, likewise
            mma_ss(tmem + C::cDP, dOnes, dDA, idSt, 1u);
            tc_commit(&bar[C::DPFULL]);
            tc_commit(&bar[C::DOEMPTY]);  // first of the two arrivals: dP^T has read dO
        }
    }
}

template <int D>
__device__ __forceinline__ void issue_grads(const BwdParams& p, const Shared& sh, const WaitCtx& w)
{
    using C = Cfg<D>;
    uint64_t* bar = sh.bar;
    const uint32_t tmem = sh.tmem;
    constexpr uint32_t idKV = idesc_bf16_f32(128, D, false, true);
    constexpr uint32_t idQ = idesc_bf16_f32(128, BQ, true, true);
    const uint64_t dQm = sdesc_sw128(smem_u32(sh.smem + C::kQ0), BQ * 128, 1024);
    const uint64_t dDOm = sdesc_sw128(smem_u32(sh.smem + C::kDO), BQ * 128, 1024);
    const uint64_t dKm = sdesc_sw128(smem_u32(sh.smem + C::kK), 16384, 1024);
    const uint64_t dDsm = sdesc_sw128(smem_u32(sh.smem + C::kDs), 16384, 1024);
    uint32_t uc = 0, n = 0;
    for (int u = blockIdx.x; u < p.total_units; u += gridDim.x) {
        Unit un = bwd_unit(p, u);
        const int T = unit_steps(p, un);
        if (T == 0)
            continue;
        if (!mbar_wait(&bar[C::KVFULL], uc & 1, w, 66))
            return;
        ++uc;
        for (int it = 0; it < T; ++it, ++n) {
            const int qs = n % C::kQStages;
            const uint32_t ph = n & 1;
            if (!mbar_wait(&bar[C::PREADY], ph, w, 63))
                return;
            // dO(n) may not have landed yet: its arrival is otherwise only
            // waited for by dP^T(n), which can be issued after this
            if (!mbar_wait(&bar[C::DOFULL], ph, w, 68))
                return;
            tc_fence_after();
            // dV += P^T dO
#pragma unroll
            for (int kk = 0; kk < BQ / 16; ++kk)
                mma_ts(tmem + C::cDV, tmem + C::cS + ptcol(kk), sdesc_add(dDOm, kk * 2048), idKV,
                       (it > 0 || kk > 0) ? 1u : 0u);
            tc_commit(&bar[C::DOEMPTY]);  // second arrival: dV has read dO
            if (!mbar_wait(&bar[C::DSREADY], ph, w, 67))
                return;
            tc_fence_after();
            // dQ^T [128 x BQ] = K^T [128 x kv] dS^T [kv x BQ], into the dP^T columns
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_ss(tmem + C::cDP, sdesc_add(dKm, kk * 2048), sdesc_add(dDsm, kk * 2048), idQ,
                       kk > 0);
            tc_commit(&bar[C::DQFULL]);
            // dK += dS^T Q, dS^T from the shared-memory tile
#pragma unroll
            for (int kk = 0; kk < BQ / 16; ++kk)
                mma_ts(tmem + C::cDK, tmem + C::cS + 32 + ptcol(kk),
                       sdesc_add(dQm, qs * C::kQTile + kk * 2048), idKV,
                       (it > 0 || kk > 0) ? 1u : 0u);
            tc_commit(&bar[C::QEMPTY + qs]);
            tc_commit(&bar[C::DKDONE]);
        }
        // all of the unit's MMAs are complete once these land: the S^T / dP^T
        // of its last step completed before its softmax, hence before its dK
        tc_commit(&bar[C::DKVFULL]);
        tc_commit(&bar[C::KVEMPTY]);
    }
}

// P^T for 32 query columns of one key row from its shifted scores, two
// columns at a time (f32x2): the tensor core already subtracted LSE/scale, so
// P = exp2((S - LSE/scale) scale log2 e).  With kMask, columns outside
// [lo, hi) (counted from the first of the 32) are not visible to this key row
// and get P = 0; a key row past the tile end is never visible.  pp receives
// the bf16 pairs.
template <bool kMask>
__device__ __forceinline__ void p_from_s(const uint32_t* sr, uint32_t* pp, uint64_t c2x2, int lo,
                                         int hi)
{
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        float a0, a1;
        f2unpack(f2mul(f2pack(__uint_as_float(sr[2 * j]), __uint_as_float(sr[2 * j + 1])), c2x2),
                 a0, a1);
        float p0 = ex2(a0), p1 = ex2(a1);
        if (kMask) {
            p0 = (2 * j >= lo && 2 * j < hi) ? p0 : 0.f;
            p1 = (2 * j + 1 >= lo && 2 * j + 1 < hi) ? p1 : 0.f;
        }
        pp[j] = pack_bf16x2(p0, p1);
    }
}

// ---------------------------------------------------------------------------
// P^T / dS^T warpgroups (warps 0-7), one thread per key row, warpgroup h on
// query columns [64 h, 64 h + 64) of each step; dK (h = 0) / dV (h = 1)
// epilogue at the end of a unit.
// ---------------------------------------------------------------------------
template <int D>
__device__ __forceinline__ void softmax_grad(const BwdParams& p, const Shared& sh,
                                             const WaitCtx& w)
{
    using C = Cfg<D>;
    uint64_t* bar = sh.bar;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = warp >> 2;                 // column half of this warpgroup
    const int r = (warp & 3) * 32 + lane;    // key row inside the unit tile (TMEM lane)
    const uint32_t tl = sh.tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t tS = tl + C::cS + 64 * h, tDP = tl + C::cDP + 64 * h;
    uint8_t* dsb = sh.smem + C::kDs + h * 16384;
    const uint32_t dsb_s = smem_u32(dsb);
    const uint64_t c2x2 = f2pack(p.scale_log2, p.scale_log2);
    // the fp32 dK / dV sums of query-blocked launches stay in L2 like dQ's
    const uint64_t keep = l2_policy_evict_last();
    uint32_t n = 0, uc = 0;
    for (int u = blockIdx.x; u < p.total_units; u += gridDim.x) {
        Unit un = bwd_unit(p, u);
        const int T = unit_steps(p, un);
        const bool kvalid = r < un.nvalid;
        const int32_t pk = kvalid ? map_pos(p.kmap[un.chunk], un.row0 + r) : 0;
        int32_t dlo, dhi;
        doc_range(p.docs, p.ndocs, pk, dlo, dhi);
        if (T > 0) {
            for (int s = 0; s < p.nq; ++s) {
                QRange qr = q_range(p, un, s);
                if (qr.i0 >= qr.i1)
                    continue;
                // query rows [qv, qe) of chunk qr.p see this key row
                const int32_t qv =
                    !kvalid ? 0x7fffffff
                            : map_count_le(p.qmap[qr.p], (p.causal ? pk : dlo) - 1);
                const int32_t qe = map_count_le(p.qmap[qr.p], dhi - 1);
                for (int i = qr.i0; i < qr.i1; ++i) {
                    for (int g = 0; g < p.G; ++g, ++n) {
                        const uint32_t ph = n & 1;
                        // tiles that see every key row take a path without
                        // any mask arithmetic
                        const bool full = (i >= qr.if0 && i < qr.if1) &&
                                          un.nvalid == kKvRows;
                        const int qbase = i * BQ + 64 * h;
                        if (!mbar_wait(&bar[C::SFULL], ph, w, 71))
                            return;
                        tc_fence_after();
                        // phase 1: P^T of the 64 columns, in two halves of 32;
                        // half c is packed into columns [16 c, 16 c + 16) of
                        // this warpgroup's 64, which half c + 1 no longer reads
                        uint32_t pp[32];
#pragma unroll
                        for (int c = 0; c < 2; ++c) {
                            uint32_t sr[32];
                            tmem_ld32(tS + 32 * c, sr);
                            tmem_ld_wait();
                            tmem_reg_fence32(sr);
                            if (full)
                                p_from_s<false>(sr, pp + 16 * c, c2x2, 0, 32);
                            else
                                p_from_s<true>(sr, pp + 16 * c, c2x2, qv - qbase - 32 * c,
                                               qe - qbase - 32 * c);
                            tmem_st16(tS + 16 * c, pp + 16 * c);
                        }
                        tmem_st_wait();
                        tc_fence_before();
                        mbar_arrive(&bar[C::PREADY]);
                        // phase 2: dS^T = P^T (dP^T - D), D already subtracted by
                        // the tensor core; P^T in bf16, as the dV product uses it
                        if (!mbar_wait(&bar[C::DPFULL], ph, w, 70))
                            return;
                        tc_fence_after();
                        // dQ^T and dK of step n - 1 have read the dS^T tile
                        // and the packed dS^T (implied by S^T(n), which
                        // was issued after dK(n - 1))
                        if (n >= 1 && !mbar_wait(&bar[C::DKDONE], (n - 1) & 1, w, 72))
                            return;
#pragma unroll
                        for (int c = 0; c < 2; ++c) {
                            uint32_t dr[32], dd[16];
                            tmem_ld32(tDP + 32 * c, dr);
                            tmem_ld_wait();
                            tmem_reg_fence32(dr);
#pragma unroll
                            for (int j = 0; j < 16; ++j) {
                                const uint32_t pj = pp[16 * c + j];
                                float d0, d1;
                                f2unpack(f2mul(f2pack(bf16lo(pj), bf16hi(pj)),
                                               f2pack(__uint_as_float(dr[2 * j]),
                                                      __uint_as_float(dr[2 * j + 1]))),
                                         d0, d1);
                                dd[j] = pack_bf16x2(d0, d1);
                            }
                            tmem_st16(tS + 32 + 16 * c, dd);
#pragma unroll
                            for (int ch = 0; ch < 4; ++ch)
                                st_shared_v4(dsb_s + sw128_offset(r, 4 * c + ch), dd[4 * ch],
                                             dd[4 * ch + 1], dd[4 * ch + 2], dd[4 * ch + 3]);
                        }
                        tmem_st_wait();
                        fence_proxy_async_smem();
                        tc_fence_before();
                        mbar_arrive(&bar[C::DSREADY]);
                    }
                }
            }
            if (!mbar_wait(&bar[C::DKVFULL], uc & 1, w, 73))
                return;
            ++uc;
            tc_fence_after();
        }
        // epilogue: warpgroup 0 stores dK (scaled), warpgroup 1 dV
        const size_t orow = (size_t)un.slice * p.Lk + (size_t)un.chunk * p.chunk_k + un.row0 + r;
        const uint32_t col = h == 0 ? C::cDK : C::cDV;
        const float mul = h == 0 ? p.scale : 1.f;
        void* outp = h == 0 ? p.dk : p.dv;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t o[32];
            if (T > 0) {
                tmem_ld32(tl + col + c0, o);
                tmem_ld_wait();
                tmem_reg_fence32(o);
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    o[e] = 0u;
            }
            if (kvalid && p.dkv_mode == 0 &&
                in_bounds(p.status, orow < (size_t)p.BHkv * p.Lk, 3, (long long)orow)) {
                uint4* dst =
                    reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(outp) + orow * D + c0);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    dst[e] = make_uint4(pack_bf16x2(__uint_as_float(o[8 * e + 0]) * mul,
                                                    __uint_as_float(o[8 * e + 1]) * mul),
                                        pack_bf16x2(__uint_as_float(o[8 * e + 2]) * mul,
                                                    __uint_as_float(o[8 * e + 3]) * mul),
                                        pack_bf16x2(__uint_as_float(o[8 * e + 4]) * mul,
                                                    __uint_as_float(o[8 * e + 5]) * mul),
                                        pack_bf16x2(__uint_as_float(o[8 * e + 6]) * mul,
                                                    __uint_as_float(o[8 * e + 7]) * mul));
            }
            if (p.dkv_mode != 0 && T > 0) {
                // fp32 accumulators shared with other units of this key tile
                // (other query blocks, other chunk-pair calls): atomic adds,
                // made row-contiguous through this warpgroup's half of the
                // dS^T tile (free once the unit's products are complete):
                // each thread stores its row's 32 values (16-byte pieces
                // XOR-swizzled by row), then each warp adds whole rows, 128
                // bytes per instruction
                float* stage = reinterpret_cast<float*>(dsb);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    st_shared_v4(dsb_s + sw128_offset(r, e),
                                 __float_as_uint(__uint_as_float(o[4 * e + 0]) * mul),
                                 __float_as_uint(__uint_as_float(o[4 * e + 1]) * mul),
                                 __float_as_uint(__uint_as_float(o[4 * e + 2]) * mul),
                                 __float_as_uint(__uint_as_float(o[4 * e + 3]) * mul));
                asm volatile("bar.sync %0, 128;" ::"r"(1 + h) : "memory");
                const int wq = warp & 3;
                const size_t rbase = (size_t)un.slice * p.Lk + (size_t)un.chunk * p.chunk_k + un.row0;
                for (int rr = wq * 32; rr < wq * 32 + 32; ++rr) {
                    if (rr >= un.nvalid ||
                        !in_bounds(p.status, rbase + rr < (size_t)p.BHkv * p.Lk, 4,
                                   (long long)(rbase + rr)))
                        break;
                    const float val = stage[rr * 32 + (((lane >> 2) ^ (rr & 7)) * 4) + (lane & 3)];
                    red_add_f32(reinterpret_cast<float*>(outp) + (rbase + rr) * D + c0 + lane, val,
                                keep);
                }
                asm volatile("bar.sync %0, 128;" ::"r"(1 + h) : "memory");
            }
        }
        // both warpgroups staged through the shared dS^T tile: neither may
        // write the next unit's dS^T before the other has finished
        if (p.dkv_mode != 0 && T > 0)
            asm volatile("bar.sync 3, 256;" ::: "memory");
        tc_fence_before();
    }
}

// ---------------------------------------------------------------------------
// dQ drain (warps 8-11): TMEM lane = feature column, columns = the step's rows
// ---------------------------------------------------------------------------
template <int D>
__device__ __forceinline__ void dq_drain(const BwdParams& p, const Shared& sh, const WaitCtx& w)
{
    using C = Cfg<D>;
    uint64_t* bar = sh.bar;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int L = (warp & 3) * 32 + lane;
    const uint32_t tl = sh.tmem + ((uint32_t)((warp & 3) * 32) << 16) + C::cDP;
    const float sc = p.scale;
    // the fp32 dQ rows are added into by every unit whose keys they see:
    // keeping them in L2 ahead of the streamed Q / dO tiles halves the
    // launch's DRAM traffic (128K: 55 -> 28 GB per 4 heads) and gains 11 %
    const uint64_t keep = l2_policy_evict_last();
    uint32_t n = 0;
    for (int u = blockIdx.x; u < p.total_units; u += gridDim.x) {
        Unit un = bwd_unit(p, u);
        if (unit_steps(p, un) == 0)
            continue;
        const int b0 = un.slice / p.Hkv, hk = un.slice % p.Hkv;
        for (int s = 0; s < p.nq; ++s) {
            QRange qr = q_range(p, un, s);
            for (int i = qr.i0; i < qr.i1; ++i) {
                for (int g = 0; g < p.G; ++g, ++n) {
                    const int slice_q = b0 * p.Hq + hk * p.G + g;
                    float* base =
                        p.dq_acc + ((size_t)slice_q * p.Lq + (size_t)qr.p * p.chunk_q) * D + L;
                    if (!mbar_wait(&bar[C::DQFULL], n & 1, w, 80))
                        return;
                    tc_fence_after();
                    uint32_t v[128];
                    tmem_ld32(tl, v);
                    tmem_ld32(tl + 32, v + 32);
                    tmem_ld32(tl + 64, v + 64);
                    tmem_ld32(tl + 96, v + 96);
                    tmem_ld_wait();
                    tmem_reg_fence32(v);
                    tmem_reg_fence32(v + 32);
                    tmem_reg_fence32(v + 64);
                    tmem_reg_fence32(v + 96);
                    tc_fence_before();
                    mbar_arrive(&bar[C::DQEMPTY]);
                    const int m0 = i * BQ;
                    const int nrow = min(BQ, p.chunk_q - m0);
                    // rows [m0, m0 + nrow) of chunk qr.p of query head slice_q
                    if (L < D &&
                        in_bounds(p.status,
                                  m0 >= 0 && nrow > 0 && qr.p < p.nq &&
                                      (size_t)slice_q * p.Lq + (size_t)qr.p * p.chunk_q + m0 +
                                              nrow <= (size_t)p.BHkv * p.G * p.Lq,
                                  5, (long long)slice_q * p.Lq + qr.p * p.chunk_q + m0)) {
                        if (nrow == BQ) {
#pragma unroll
                            for (int c = 0; c < BQ; ++c)
                                red_add_f32(base + (size_t)(m0 + c) * D, __uint_as_float(v[c]) * sc,
                                            keep);
                        } else {
#pragma unroll
                            for (int c = 0; c < BQ; ++c)
                                if (c < nrow)
                                    red_add_f32(base + (size_t)(m0 + c) * D,
                                                __uint_as_float(v[c]) * sc, keep);
                        }
                    }
                }
            }
        }
    }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                    const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmdo,
                    const __grid_constant__ CUtensorMap tmal,
                    const __grid_constant__ CUtensorMap tmad, const __grid_constant__ BwdParams p)
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
        mbar_init(&bar[C::KVFULL], 1);
        mbar_init(&bar[C::KVEMPTY], 1);
        for (int s = 0; s < C::kQStages; ++s) {
            mbar_init(&bar[C::QFULL + s], 1);
            mbar_init(&bar[C::QEMPTY + s], 1);
        }
        mbar_init(&bar[C::DOFULL], 1);
        mbar_init(&bar[C::DOEMPTY], 2);
        mbar_init(&bar[C::SFULL], 1);
        mbar_init(&bar[C::DPFULL], 1);
        mbar_init(&bar[C::PREADY], 256);
        mbar_init(&bar[C::DSREADY], 256);
        mbar_init(&bar[C::DQFULL], 1);
        mbar_init(&bar[C::DQEMPTY], 128);
        mbar_init(&bar[C::DKVFULL], 1);
        mbar_init(&bar[C::DKDONE], 1);
        fence_barrier_init();
    }
    {
        // the ones tile: every 32-byte row holds 1.0 at K positions 0, 1, 8
        // and 9; its two 16-byte halves are equal, so the swizzle leaves it
        // as is
        uint4* ones = (uint4*)(smem + C::kOnes);
        for (int i = threadIdx.x; i < 128 * 2; i += blockDim.x)
            ones[i] = make_uint4(0x3F803F80u, 0u, 0u, 0u);
        fence_proxy_async_smem();
    }
    if (D < 128) {
        // zero the K tile's padding columns once (TMA never writes them)
        uint4* pad = (uint4*)(smem + C::kK + 16384);
        for (int i = threadIdx.x; i < 16384 / 16; i += blockDim.x)
            pad[i] = make_uint4(0u, 0u, 0u, 0u);
        fence_proxy_async_smem();
    }
    if (warp == kWarpMma) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const Shared sh{smem, bar, abort_flag, *tmem_slot};

    if (warp >= 12) {
        reg_dealloc<kRegsCtl>();
        if (warp == kWarpProducer) {
            producer<D>(p, sh, wctx, &tmq, &tmk, &tmv, &tmdo, &tmal, &tmad);
            if (lane == 0 && *abort_flag) {
                // give copies already issued a bounded chance to land
                const uint64_t t0 = globaltimer_ns();
                while (globaltimer_ns() - t0 < 2000000ull) {
                }
            }
        } else if (warp == kWarpMma && lane == 0) {
            issue_grads<D>(p, sh, wctx);
        } else if (warp == kWarpMmaS && lane == 0) {
            issue_products<D>(p, sh, wctx);
        }
    } else if (warp >= 8) {
        reg_alloc<kRegsDrain>();
        dq_drain<D>(p, sh, wctx);
    } else {
        reg_alloc<kRegsSoft>();
        softmax_grad<D>(p, sh, wctx);
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(sh.tmem, 512);
    }
}

}  // namespace bwd

cudaError_t launch_attn_bwd(int d, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& tdo,
                            const CUtensorMap& tal, const CUtensorMap& tad, const BwdParams& p,
                            int grid, cudaStream_t stream)
{
    if (d == 128) {
        constexpr int smem = bwd::Cfg<128>::kSmem;
        cudaError_t e = cudaFuncSetAttribute(bwd::attn_bwd_kernel<128>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess)
            return e;
        bwd::attn_bwd_kernel<128><<<grid, bwd::kThreads, smem, stream>>>(tq, tk, tv, tdo, tal, tad, p);
    } else {
        constexpr int smem = bwd::Cfg<64>::kSmem;
        cudaError_t e = cudaFuncSetAttribute(bwd::attn_bwd_kernel<64>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess)
            return e;
        bwd::attn_bwd_kernel<64><<<grid, bwd::kThreads, smem, stream>>>(tq, tk, tv, tdo, tal, tad, p);
    }
    return cudaGetLastError();
}

int bwd_rows_per_unit() { return bwd::kKvRows; }
int bwd_query_rows_per_step() { return bwd::BQ; }

}  // namespace dfa
