// dfa_params.h -- plain-data structures shared by the host launchers and the
// kernels: per-chunk position maps, the query-row work units of a launch, and
// the kernel parameter blocks.
//
// A launch sees the sequence as nq query chunks and nkv key/value chunks of
// fixed row counts, each chunk carrying a monotone map from its local rows to
// global token positions.  Whole attention is one chunk with the identity
// map; a worker-major (permuted) layout is P chunks with the partition's maps;
// a single chunk pair is one query chunk and one key/value chunk.
#pragma once

#include <cstdint>

#ifdef __CUDACC__
#define DFA_HD __host__ __device__ __forceinline__
#else
#define DFA_HD inline
#endif

namespace dfa {

constexpr int kMaxChunks = 32;  // chunks per side of one launch
constexpr int kMaxSegs = 64;    // query segments of one launch

// Monotone map of a chunk's local rows to global positions.  Rows [0, len0)
// form segment 0, rows [len0, len0 + len1) segment 1; row m' of a segment has
// position base + (m' / blk) * blk_stride + m' % blk.
struct DevMap {
    int32_t len0, len1;
    int32_t base0, base1;
    int32_t blk, blk_stride;
};

DFA_HD int32_t map_pos(const DevMap& m, int32_t r)
{
    int32_t b, x;
    if (r < m.len0) {
        b = m.base0;
        x = r;
    } else {
        b = m.base1;
        x = r - m.len0;
    }
    if (m.blk == 1)
        return b + x * m.blk_stride;
    return b + (x / m.blk) * m.blk_stride + (x % m.blk);
}

// Rows of one segment whose position is <= x.  32-bit arithmetic (positions
// lie in [0, 2^31), base >= 0 for a non-empty segment) and no division for a
// run of consecutive positions: the kernels evaluate this at every chunk of
// every work unit, on the path between tensor-core steps.
DFA_HD int32_t seg_count_le(int32_t base, int32_t len, int32_t blk, int32_t stride, int32_t x)
{
    if (len <= 0 || x < base)
        return 0;
    const int32_t dlt = x - base;
    if (blk == stride)
        return dlt < len ? dlt + 1 : len;
    const int32_t runs = dlt / stride;
    const int32_t off = dlt - runs * stride;
    const int32_t c = runs * blk + (off < blk ? off + 1 : blk);
    return c < len ? c : len;
}

// Number of rows of the chunk whose position is <= x.  Because positions
// increase along the chunk, these rows are exactly rows [0, count).
DFA_HD int32_t map_count_le(const DevMap& m, int32_t x)
{
    return seg_count_le(m.base0, m.len0, m.blk, m.blk_stride, x) +
           seg_count_le(m.base1, m.len1, m.blk, m.blk_stride, x);
}

DFA_HD int32_t ceil_div(int32_t a, int32_t b) { return (a + b - 1) / b; }

// Packed documents: positions [bounds[t], bounds[t+1]), t < ndocs, form
// document t.  doc_range gives the document [lo, hi) of position x; without
// documents (ndocs = 0) it is the whole line.
constexpr int32_t kPosLo = INT32_MIN + 2, kPosHi = INT32_MAX - 1;

DFA_HD void doc_range(const int64_t* bounds, int32_t ndocs, int32_t x, int32_t& lo, int32_t& hi)
{
    if (ndocs <= 0) {
        lo = kPosLo;
        hi = kPosHi;
        return;
    }
    int32_t a = 0, c = ndocs;  // largest t with bounds[t] <= x
    while (c - a > 1) {
        const int32_t mid = (a + c) / 2;
        if (bounds[mid] <= x)
            a = mid;
        else
            c = mid;
    }
    lo = (int32_t)bounds[a];
    hi = (int32_t)bounds[a + 1];
}

// Work units.  The rows of every chunk are cut into segments (runs of rows
// inside one map segment) and each segment into units of `rows_per_unit`
// rows; units are replicated over the BH (batch x head) slices.  Inside a
// slice, units are issued longest-first: by segment in the order given (the
// host sorts segments by position), or, with tile_major, round by round across
// equal-length segments.  Slices are issued one after another (all units of
// slice 0, then slice 1, ...), so that the CTAs running at the same time share
// one head's K/V (forward) or Q/dO/dQ rows (backward) in L2.
struct UnitTable {
    int32_t nsegs;
    int32_t tile_major;
    int32_t units_per_slice;  // units per BH slice
    int32_t rounds;           // tile_major: units per segment
    int32_t seg_chunk[kMaxSegs];
    int32_t seg_start[kMaxSegs];
    int32_t seg_len[kMaxSegs];
    int32_t seg_prefix[kMaxSegs + 1];  // cumulative units before each segment
};

struct Unit {
    int32_t slice;   // BH index (b * H + h) of the side the units are cut from
    int32_t chunk;   // chunk index
    int32_t row0;    // first local row of the unit inside the chunk
    int32_t nvalid;  // rows of the unit inside the segment (<= rows_per_unit)
    int32_t qblk;    // backward: query block of the unit (0 without blocking)
};

DFA_HD Unit decode_unit(const UnitTable& t, int32_t nslices, int32_t rows_per_unit, int32_t u,
                        bool reverse)
{
    Unit r;
    (void)nslices;
    int32_t rank = u % t.units_per_slice;
    r.slice = u / t.units_per_slice;
    int32_t seg, k;
    if (t.tile_major) {
        seg = rank % t.nsegs;
        k = rank / t.nsegs;
        if (!reverse)
            k = t.rounds - 1 - k;
    } else {
        seg = 0;
        while (seg + 1 < t.nsegs && rank >= t.seg_prefix[seg + 1])
            ++seg;
        int32_t nu = t.seg_prefix[seg + 1] - t.seg_prefix[seg];
        k = rank - t.seg_prefix[seg];
        if (!reverse)
            k = nu - 1 - k;
    }
    r.chunk = t.seg_chunk[seg];
    r.row0 = t.seg_start[seg] + k * rows_per_unit;
    int32_t rem = t.seg_start[seg] + t.seg_len[seg] - r.row0;
    r.nvalid = rem < rows_per_unit ? rem : rows_per_unit;
    r.qblk = 0;
    return r;
}

struct DevStatus;

// Permute parameters: rows of worker-major order r = p n + m hold natural row
// map[p](m).
struct PermuteParams {
    int64_t heads;
    int32_t N, n, P;
    int32_t row_vecs;
    int32_t inverse;
    DevMap map[kMaxChunks];
};

// Split-KV decoding: T query tokens per sequence against L cached keys.
struct DecodeParams {
    int32_t B, Hq, Hkv, G, T;
    int32_t L;                   // cached keys per (b, kv head)
    int32_t split_len;           // keys per split (multiple of 64)
    int32_t causal;
    int64_t q_pos0;              // position of query token 0; key j is at position j
    float scale_log2;            // scale * log2(e)
    const void* q;               // [B, Hq, T, d] bf16
    const void* k;               // [B, Hkv, L, d] bf16
    const void* v;
    float* o_part;               // [splits, B*Hq*T, d] fp32
    float* lse_part;             // [splits, B*Hq*T] fp32
};

// Rotary embedding fused into the permute: theta[t] = base^(-2t/d) for the
// feature pairs (2t, 2t+1), t < d/2.
struct RopeParams {
    PermuteParams perm;
    int32_t d;
    double theta[64];
};

// Forward kernel parameters.
struct FwdParams {
    int32_t BH, Hq, Hkv, G;
    int32_t Lq, Lk;              // rows per head slice in q / kv storage
    int32_t nq, nkv;             // chunks per side
    int32_t chunk_q, chunk_k;    // rows per chunk
    int32_t causal;
    float scale, scale_log2;
    int32_t total_units;
    int32_t o_fp32;
    int32_t ndocs;               // packed documents (0: none)
    const int64_t* docs;         // [ndocs + 1] cumulative positions (device)
    UnitTable units;
    DevMap qmap[kMaxChunks];
    DevMap kmap[kMaxChunks];
    void* o;
    float* lse;
    DevStatus* status;
    uint64_t timeout_ns;
};

// Backward main-kernel parameters.  Units are key/value tiles.
struct BwdParams {
    int32_t BHkv, Hq, Hkv, G;
    int32_t Lq, Lk;
    int32_t nq, nkv;
    int32_t chunk_q, chunk_k;
    int32_t causal;
    float scale, scale_log2;
    int32_t total_units;
    int32_t dkv_mode;            // 0: write bf16 dK/dV; 1: add into fp32 (atomic)
    int32_t nqblk;               // query blocks per key tile (1: no blocking)
    int32_t qblk_tiles;          // query tiles per block and chunk
    int32_t ndocs;               // packed documents (0: none)
    const int64_t* docs;         // [ndocs + 1] cumulative positions (device)
    UnitTable units;
    DevMap qmap[kMaxChunks];
    DevMap kmap[kMaxChunks];
    float* dq_acc;               // [BHq, Lq, d] fp32, scaled
    void* dk;                    // [BHkv, Lk, d]
    void* dv;
    DevStatus* status;
    uint64_t timeout_ns;
};

}  // namespace dfa
