// dfa_api.cu -- the C ABI of libdfa (include/dfa.h): argument validation,
// partition maps, work-unit tables, TMA tensor maps, kernel launches, the
// host-side ring schedule, and status reporting.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "../../include/dfa.h"
#include "dfa_launch.h"
#include "dfa_params.h"
#include "dfa_ptx.cuh"

using namespace dfa;

namespace {

thread_local char g_last_error[512] = "";

dfa_status fail(dfa_status s, const char* fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return s;
}

dfa_status cuda_fail(cudaError_t e, const char* what)
{
    return fail(DFA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

constexpr size_t kStatusBytes = 256;
constexpr uint64_t kDefaultTimeoutNs = 4000000000ull;  // 4 s per wait

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

int num_sms()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return 1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 1;
    return n > 0 ? n : 1;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// ----------------------------------------------------------------------------
// position maps
// ----------------------------------------------------------------------------
dfa_status check_map(const dfa_pos_map& m, int64_t L, const char* name)
{
    if (m.nseg != 1 && m.nseg != 2)
        return fail(DFA_ERR_INVALID_ARG, "%s: nseg must be 1 or 2", name);
    int64_t l1 = m.nseg == 2 ? m.len[1] : 0;
    if (m.len[0] < 0 || l1 < 0 || m.len[0] + l1 != L)
        return fail(DFA_ERR_INVALID_ARG, "%s: segment lengths do not add up to %lld", name,
                    (long long)L);
    if (m.blk < 1 || m.blk_stride < m.blk)
        return fail(DFA_ERR_UNSUPPORTED, "%s: need blk >= 1 and blk_stride >= blk", name);
    for (int t = 0; t < m.nseg; ++t) {
        int64_t len = m.len[t];
        if (len == 0)
            continue;
        int64_t last = m.base[t] + ((len - 1) / m.blk) * m.blk_stride + (len - 1) % m.blk;
        if (m.base[t] < 0 || last >= INT32_MAX)
            return fail(DFA_ERR_UNSUPPORTED, "%s: positions must lie in [0, 2^31)", name);
        if (t == 1 && m.len[0] > 0) {
            int64_t l0 = m.len[0];
            int64_t last0 = m.base[0] + ((l0 - 1) / m.blk) * m.blk_stride + (l0 - 1) % m.blk;
            if (m.base[1] <= last0)
                return fail(DFA_ERR_UNSUPPORTED,
                            "%s: positions must increase along the chunk", name);
        }
    }
    return DFA_OK;
}

DevMap to_dev(const dfa_pos_map& m)
{
    DevMap d;
    d.len0 = (int32_t)m.len[0];
    d.len1 = m.nseg == 2 ? (int32_t)m.len[1] : 0;
    d.base0 = (int32_t)m.base[0];
    d.base1 = m.nseg == 2 ? (int32_t)m.base[1] : 0;
    d.blk = (int32_t)m.blk;
    d.blk_stride = (int32_t)m.blk_stride;
    return d;
}

dfa_pos_map identity_map(int64_t L)
{
    dfa_pos_map m{};
    m.nseg = 1;
    m.len[0] = L;
    m.base[0] = 0;
    m.blk = 1;
    m.blk_stride = 1;
    return m;
}

dfa_status check_desc(const dfa_attn_desc* d, bool need_partition)
{
    if (!d)
        return fail(DFA_ERR_INVALID_ARG, "desc is NULL");
    if (d->B < 1 || d->Hq < 1 || d->Hkv < 1 || d->N < 1)
        return fail(DFA_ERR_INVALID_ARG, "B, Hq, Hkv, N must be positive");
    if (d->Hq % d->Hkv != 0)
        return fail(DFA_ERR_INVALID_ARG, "Hq (%d) must be a multiple of Hkv (%d)", d->Hq, d->Hkv);
    if (d->d != 64 && d->d != 128)
        return fail(DFA_ERR_UNSUPPORTED, "head dimension %d not supported (64 or 128)", d->d);
    if (d->N >= (int64_t)INT32_MAX - 1024)
        return fail(DFA_ERR_UNSUPPORTED, "N too large");
    if ((int64_t)d->B * d->Hq >= INT32_MAX / 4)
        return fail(DFA_ERR_UNSUPPORTED, "B*Hq too large");
    if (!(d->scale > 0.f) || !std::isfinite(d->scale))
        return fail(DFA_ERR_INVALID_ARG, "scale must be positive and finite");
    if (d->causal != 0 && d->causal != 1)
        return fail(DFA_ERR_INVALID_ARG, "causal must be 0 or 1");
    if (d->ndocs < 0 || (d->ndocs > 0 && !d->doc_bounds))
        return fail(DFA_ERR_INVALID_ARG, "ndocs must be >= 0, with doc_bounds when > 0");
    if (need_partition) {
        if (d->P < 1 || d->P > kMaxChunks)
            return fail(DFA_ERR_UNSUPPORTED, "P must be in [1, %d]", kMaxChunks);
        if (d->N % d->P != 0)
            return fail(DFA_ERR_INVALID_ARG, "N %% P != 0");
        if (d->partition < 0 || d->partition > 2)
            return fail(DFA_ERR_INVALID_ARG, "unknown partition %d", d->partition);
        if (d->partition == DFA_PART_BALANCED && d->N % (2 * (int64_t)d->P) != 0)
            return fail(DFA_ERR_INVALID_ARG, "balanced partition needs N %% 2P == 0");
        if (d->partition == DFA_PART_STRIPED &&
            (d->stripe < 1 || d->N % ((int64_t)d->stripe * d->P) != 0))
            return fail(DFA_ERR_INVALID_ARG, "striped partition needs N %% (stripe*P) == 0");
    }
    return DFA_OK;
}

dfa_pos_map partition_map(const dfa_attn_desc& d, int p)
{
    const int64_t n = d.N / d.P;
    dfa_pos_map m{};
    m.blk = 1;
    m.blk_stride = 1;
    if (d.partition == DFA_PART_CONTIGUOUS || d.P == 1) {
        m.nseg = 1;
        m.len[0] = n;
        m.base[0] = (int64_t)p * n;
    } else if (d.partition == DFA_PART_BALANCED) {
        const int64_t c = d.N / (2 * (int64_t)d.P);
        m.nseg = 2;
        m.len[0] = c;
        m.len[1] = c;
        m.base[0] = (int64_t)p * c;
        m.base[1] = (int64_t)(2 * d.P - 1 - p) * c;
    } else {
        const int64_t s = d.stripe;
        m.nseg = 1;
        m.len[0] = n;
        m.base[0] = (int64_t)p * s;
        m.blk = s;
        m.blk_stride = (int64_t)d.P * s;
    }
    return m;
}

// Launch layout of a (possibly permuted) whole sequence: contiguous order is
// one identity chunk; folded / striped worker-major order is P chunks.
int layout_chunks(const dfa_attn_desc& d)
{
    return (d.P == 1 || d.partition == DFA_PART_CONTIGUOUS) ? 1 : d.P;
}

// ----------------------------------------------------------------------------
// work-unit tables
// ----------------------------------------------------------------------------
struct Seg {
    int chunk, start, len;
    int64_t key;  // position of the segment's first row
};

// descending = true: segments with the highest positions first (forward,
// query rows late in the sequence have the most keys); false: lowest first
// (backward, key rows early in the sequence have the most queries).
UnitTable build_units(const std::vector<dfa_pos_map>& maps, int rows_per_unit, bool descending)
{
    std::vector<Seg> segs;
    bool interleaved = false;
    for (int c = 0; c < (int)maps.size(); ++c) {
        const dfa_pos_map& m = maps[c];
        int64_t start = 0;
        for (int t = 0; t < m.nseg; ++t) {
            if (m.len[t] > 0)
                segs.push_back({c, (int)start, (int)m.len[t], m.base[t]});
            start += m.len[t];
        }
        if (m.blk_stride > m.blk)
            interleaved = true;
    }
    std::stable_sort(segs.begin(), segs.end(), [&](const Seg& a, const Seg& b) {
        return descending ? a.key > b.key : a.key < b.key;
    });
    UnitTable t{};
    t.nsegs = (int)segs.size();
    bool equal = true;
    for (auto& s : segs)
        equal = equal && s.len == segs[0].len;
    t.tile_major = (interleaved && equal && t.nsegs > 1) ? 1 : 0;
    t.seg_prefix[0] = 0;
    for (int i = 0; i < t.nsegs; ++i) {
        t.seg_chunk[i] = segs[i].chunk;
        t.seg_start[i] = segs[i].start;
        t.seg_len[i] = segs[i].len;
        t.seg_prefix[i + 1] = t.seg_prefix[i] + (segs[i].len + rows_per_unit - 1) / rows_per_unit;
    }
    t.units_per_slice = t.seg_prefix[t.nsegs];
    t.rounds = t.nsegs > 0 ? (segs[0].len + rows_per_unit - 1) / rows_per_unit : 0;
    return t;
}

// ----------------------------------------------------------------------------
// TMA tensor maps: [slices][rows][d] bf16, box 64 columns x box_rows rows,
// 128-byte swizzle, zero fill outside the tensor.
// ----------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
    }
    return fn;
}

dfa_status make_tmap(CUtensorMap* out, const void* ptr, int64_t slices, int64_t rows, int d,
                     int box_rows, const char* name)
{
    auto fn = encode_fn();
    if (!fn)
        return fail(DFA_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)rows, (cuuint64_t)slices};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)rows * d * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = fn(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims,
                    strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(DFA_ERR_CUDA, "tensor map for %s failed (CUresult %d)", name, (int)r);
    return DFA_OK;
}

// The backward's per-row records: [slices, rows, 16] bf16 (32 bytes a row),
// loaded 64 rows at a time with a 32-byte swizzle.
dfa_status make_tmap_aug(CUtensorMap* out, const void* ptr, int64_t slices, int64_t rows,
                         int box_rows, const char* name)
{
    auto fn = encode_fn();
    if (!fn)
        return fail(DFA_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    cuuint64_t dims[3] = {16, (cuuint64_t)rows, (cuuint64_t)slices};
    cuuint64_t strides[2] = {(cuuint64_t)kAugRowBytes, (cuuint64_t)rows * kAugRowBytes};
    cuuint32_t box[3] = {16, (cuuint32_t)box_rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = fn(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims,
                    strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(DFA_ERR_CUDA, "tensor map for %s failed (CUresult %d)", name, (int)r);
    return DFA_OK;
}

DevStatus* status_word(void* ws) { return reinterpret_cast<DevStatus*>(ws); }

dfa_status check_ws(void* ws, size_t have, size_t need)
{
    if (!ws)
        return fail(DFA_ERR_WORKSPACE, "workspace is NULL");
    if (((uintptr_t)ws & 255u) != 0)
        return fail(DFA_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    if (have < need)
        return fail(DFA_ERR_WORKSPACE, "workspace too small: %zu < %zu", have, need);
    return DFA_OK;
}

// ----------------------------------------------------------------------------
// forward / backward launches over a layout of nq query chunks and nkv kv
// chunks (shared by the whole-sequence and chunk-pair calls)
// ----------------------------------------------------------------------------
// When a key/value head's query rows -- N rows for each of its G query
// heads -- exceed kBwdBlockAbove, the backward cuts the query side into
// blocks (the same local tile range in every query chunk) of 65536 / G rows
// per head (at least 8192), so that the units running at one time share one
// block's Q, dO and dQ rows of every head of the group (about 64 MB) in L2;
// dK and dV are then summed over the blocks in fp32.  Every block pass reads
// and writes those fp32 sums, so fewer blocks cost less DRAM traffic (and
// power under the 1.4 kW cap).  Measured on GB300 (backward TFLOP/s):
// Llama-7B 128K, 32 heads: no blocks 1033 (striped and folded alike),
// 64K-row blocks 1027 / 994, 32K-row blocks 983 / 906;  512K, 8 heads
// (folded): 64K blocks 1013, 128K blocks 990, 32K blocks 927;  grouped-query
// 64K (G = 4, query heads innermost in a unit): 16K blocks 922, 32K 889,
// none 805.
constexpr int64_t kBwdBlockAbove = 131072;

bool bwd_blocked(int64_t q_rows_per_head, int G) { return q_rows_per_head * G > kBwdBlockAbove; }

int64_t bwd_block_rows(int G) { return std::max<int64_t>(8192, 65536 / std::max(1, G)); }

struct Layout {
    std::vector<dfa_pos_map> qmaps, kmaps;
    int64_t chunk_q, chunk_k;
};

dfa_status run_fwd(const dfa_attn_desc& d, const Layout& lay, const void* q, const void* k,
                   const void* v, void* o, float* lse, int o_fp32, void* ws, cudaStream_t stream)
{
    const int64_t Lq = lay.chunk_q * (int64_t)lay.qmaps.size();
    const int64_t Lk = lay.chunk_k * (int64_t)lay.kmaps.size();
    FwdParams p;
    memset(&p, 0, sizeof p);
    p.BH = d.B * d.Hq;
    p.Hq = d.Hq;
    p.Hkv = d.Hkv;
    p.G = d.Hq / d.Hkv;
    p.Lq = (int32_t)Lq;
    p.Lk = (int32_t)Lk;
    p.nq = (int32_t)lay.qmaps.size();
    p.nkv = (int32_t)lay.kmaps.size();
    p.chunk_q = (int32_t)lay.chunk_q;
    p.chunk_k = (int32_t)lay.chunk_k;
    p.causal = d.causal;
    p.scale = d.scale;
    p.scale_log2 = d.scale * 1.4426950408889634f;
    p.o_fp32 = o_fp32;
    p.ndocs = d.ndocs;
    p.docs = d.doc_bounds;
    p.units = build_units(lay.qmaps, fwd_rows_per_unit(), true);
    p.total_units = p.units.units_per_slice * p.BH;
    for (size_t i = 0; i < lay.qmaps.size(); ++i)
        p.qmap[i] = to_dev(lay.qmaps[i]);
    for (size_t i = 0; i < lay.kmaps.size(); ++i)
        p.kmap[i] = to_dev(lay.kmaps[i]);
    p.o = o;
    p.lse = lse;
    p.status = status_word(ws);
    p.timeout_ns = kDefaultTimeoutNs;
    if (p.total_units == 0)
        return DFA_OK;
    CUtensorMap tq, tk, tv;
    dfa_status s;
    if ((s = make_tmap(&tq, q, p.BH, Lq, d.d, 128, "q")) != DFA_OK)
        return s;
    if ((s = make_tmap(&tk, k, (int64_t)d.B * d.Hkv, Lk, d.d, 128, "k")) != DFA_OK)
        return s;
    if ((s = make_tmap(&tv, v, (int64_t)d.B * d.Hkv, Lk, d.d, 128, "v")) != DFA_OK)
        return s;
    const int grid = std::min(p.total_units, num_sms());
    cudaError_t e = launch_attn_fwd(d.d, tq, tk, tv, p, grid, stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "attention forward launch");
    return DFA_OK;
}

dfa_status run_bwd_main(const dfa_attn_desc& d, const Layout& lay, const void* q, const void* k,
                        const void* v, const void* dout, const void* aug_lse,
                        const void* aug_delta, float* dq_acc, void* dk, void* dv, int dkv_mode,
                        void* ws, cudaStream_t stream)
{
    const int64_t Lq = lay.chunk_q * (int64_t)lay.qmaps.size();
    const int64_t Lk = lay.chunk_k * (int64_t)lay.kmaps.size();
    BwdParams p;
    memset(&p, 0, sizeof p);
    p.BHkv = d.B * d.Hkv;
    p.Hq = d.Hq;
    p.Hkv = d.Hkv;
    p.G = d.Hq / d.Hkv;
    p.Lq = (int32_t)Lq;
    p.Lk = (int32_t)Lk;
    p.nq = (int32_t)lay.qmaps.size();
    p.nkv = (int32_t)lay.kmaps.size();
    p.chunk_q = (int32_t)lay.chunk_q;
    p.chunk_k = (int32_t)lay.chunk_k;
    p.causal = d.causal;
    p.scale = d.scale;
    p.scale_log2 = d.scale * 1.4426950408889634f;
    p.dkv_mode = dkv_mode;
    p.ndocs = d.ndocs;
    p.docs = d.doc_bounds;
    p.units = build_units(lay.kmaps, bwd_rows_per_unit(), false);
    const int bq = bwd_query_rows_per_step();
    const int64_t nqt = (lay.chunk_q + bq - 1) / bq;
    p.nqblk = 1;
    p.qblk_tiles = (int32_t)nqt;
    if (bwd_blocked(Lq, d.Hq / d.Hkv)) {
        const int64_t rows_per_chunk =
            std::max<int64_t>(bq, bwd_block_rows(d.Hq / d.Hkv) / (int64_t)lay.qmaps.size());
        p.qblk_tiles = (int32_t)std::max<int64_t>(1, rows_per_chunk / bq);
        p.nqblk = (int32_t)((nqt + p.qblk_tiles - 1) / p.qblk_tiles);
    }
    if ((int64_t)p.units.units_per_slice * p.BHkv * p.nqblk >= INT32_MAX)
        return fail(DFA_ERR_UNSUPPORTED, "too many backward work units");
    p.total_units = p.units.units_per_slice * p.BHkv * p.nqblk;
    for (size_t i = 0; i < lay.qmaps.size(); ++i)
        p.qmap[i] = to_dev(lay.qmaps[i]);
    for (size_t i = 0; i < lay.kmaps.size(); ++i)
        p.kmap[i] = to_dev(lay.kmaps[i]);
    p.dq_acc = dq_acc;
    p.dk = dk;
    p.dv = dv;
    p.status = status_word(ws);
    p.timeout_ns = kDefaultTimeoutNs;
    if (p.total_units == 0)
        return DFA_OK;
    CUtensorMap tq, tk, tv, tdo, tal, tad;
    dfa_status s;
    const int64_t BHq = (int64_t)d.B * d.Hq, BHkv = (int64_t)d.B * d.Hkv;
    if ((s = make_tmap(&tq, q, BHq, Lq, d.d, bq, "q")) != DFA_OK)
        return s;
    if ((s = make_tmap_aug(&tal, aug_lse, BHq, Lq, bq, "LSE records")) != DFA_OK)
        return s;
    if ((s = make_tmap_aug(&tad, aug_delta, BHq, Lq, bq, "D records")) != DFA_OK)
        return s;
    if ((s = make_tmap(&tdo, dout, BHq, Lq, d.d, bq, "dout")) != DFA_OK)
        return s;
    if ((s = make_tmap(&tk, k, BHkv, Lk, d.d, 128, "k")) != DFA_OK)
        return s;
    if ((s = make_tmap(&tv, v, BHkv, Lk, d.d, 128, "v")) != DFA_OK)
        return s;
    const int grid = std::min(p.total_units, num_sms());
    cudaError_t e = launch_attn_bwd(d.d, tq, tk, tv, tdo, tal, tad, p, grid, stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "attention backward launch");
    return DFA_OK;
}

Layout whole_layout(const dfa_attn_desc& d)
{
    Layout lay;
    const int nc = layout_chunks(d);
    if (nc == 1) {
        lay.qmaps.push_back(identity_map(d.N));
        lay.chunk_q = d.N;
    } else {
        for (int p = 0; p < nc; ++p)
            lay.qmaps.push_back(partition_map(d, p));
        lay.chunk_q = d.N / d.P;
    }
    lay.kmaps = lay.qmaps;
    lay.chunk_k = lay.chunk_q;
    return lay;
}

dfa_status check_ptrs(std::initializer_list<const void*> ps)
{
    for (const void* p : ps) {
        if (!p)
            return fail(DFA_ERR_INVALID_ARG, "a tensor pointer is NULL");
        if (!aligned16(p))
            return fail(DFA_ERR_UNSUPPORTED, "tensor pointers must be 16-byte aligned");
    }
    return DFA_OK;
}

// Backward workspace: status word, fp32 dQ accumulator, -LSE/scale and -D
// records (32 bytes a row each), and with query blocking fp32 dK and dV.
size_t bwd_ws_bytes(const dfa_attn_desc& d)
{
    const size_t rows = (size_t)d.B * d.Hq * (size_t)d.N;
    const size_t kv = (size_t)d.B * d.Hkv * (size_t)d.N * d.d * 4;
    return kStatusBytes + align256(rows * d.d * 4) + 2 * align256(rows * kAugRowBytes) +
           (bwd_blocked(d.N, d.Hq / d.Hkv) ? 2 * align256(kv) : 0);
}

}  // namespace

namespace dfa {
// Record the calling thread's last-error text (used by other translation units).
dfa_status set_error(dfa_status s, const char* fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return s;
}
}  // namespace dfa

// ============================================================================
// C ABI
// ============================================================================
extern "C" {

const char* dfa_status_string(dfa_status s)
{
    switch (s) {
    case DFA_OK:
        return "ok";
    case DFA_ERR_INVALID_ARG:
        return "invalid argument";
    case DFA_ERR_UNSUPPORTED:
        return "unsupported";
    case DFA_ERR_WORKSPACE:
        return "workspace missing or too small";
    case DFA_ERR_CUDA:
        return "CUDA error";
    case DFA_ERR_TIMEOUT:
        return "device wait timed out";
    case DFA_ERR_BOUNDS:
        return "device index out of bounds (bounds-checking build)";
    }
    return "unknown status";
}

const char* dfa_last_error(void) { return g_last_error; }

int32_t dfa_version(void) { return 1; }

size_t dfa_workspace_size(const dfa_attn_desc* desc, int32_t op)
{
    if (check_desc(desc, op == DFA_OP_FWD || op == DFA_OP_BWD || op == DFA_OP_RING_FWD) != DFA_OK)
        return 0;
    switch (op) {
    case DFA_OP_FWD:
    case DFA_OP_CHUNK_FWD:
        return kStatusBytes;
    case DFA_OP_BWD:
        return bwd_ws_bytes(*desc);
    case DFA_OP_RING_FWD: {
        const size_t rows = (size_t)desc->B * desc->Hq * (size_t)(desc->N / desc->P);
        return kStatusBytes + align256(rows * desc->d * 4) + align256(rows * 4);
    }
    case DFA_OP_CHUNK_BWD:
        return kStatusBytes +
               2 * align256((size_t)desc->B * desc->Hq * (size_t)desc->N * kAugRowBytes);
    }
    return 0;
}

dfa_status dfa_partition_map(const dfa_attn_desc* desc, int32_t p, dfa_pos_map* out)
{
    dfa_status s = check_desc(desc, true);
    if (s != DFA_OK)
        return s;
    if (!out || p < 0 || p >= desc->P)
        return fail(DFA_ERR_INVALID_ARG, "bad worker index or NULL output");
    *out = partition_map(*desc, p);
    return DFA_OK;
}

dfa_status dfa_attn_fwd(const dfa_attn_desc* desc, const void* q, const void* k, const void* v,
                        void* o, float* lse, void* ws, size_t ws_bytes, void* stream)
{
    dfa_status s = check_desc(desc, true);
    if (s != DFA_OK)
        return s;
    if ((s = check_ptrs({q, k, v, o})) != DFA_OK)
        return s;
    if (!lse)
        return fail(DFA_ERR_INVALID_ARG, "lse is NULL");
    if ((s = check_ws(ws, ws_bytes, kStatusBytes)) != DFA_OK)
        return s;
    return run_fwd(*desc, whole_layout(*desc), q, k, v, o, lse, desc->o_fp32, ws,
                   (cudaStream_t)stream);
}

dfa_status dfa_chunk_fwd(const dfa_attn_desc* desc, const dfa_chunk_pair* pair, int64_t Lq,
                         int64_t Lk, const void* q, const void* k, const void* v, float* o_part,
                         float* lse_part, void* ws, size_t ws_bytes, void* stream)
{
    dfa_status s = check_desc(desc, false);
    if (s != DFA_OK)
        return s;
    if (!pair)
        return fail(DFA_ERR_INVALID_ARG, "pair is NULL");
    if (Lq < 1 || Lk < 1 || Lq >= INT32_MAX / 2 || Lk >= INT32_MAX / 2)
        return fail(DFA_ERR_INVALID_ARG, "chunk lengths must be in [1, 2^30)");
    if ((s = check_map(pair->q, Lq, "pair.q")) != DFA_OK)
        return s;
    if ((s = check_map(pair->kv, Lk, "pair.kv")) != DFA_OK)
        return s;
    if ((s = check_ptrs({q, k, v, o_part})) != DFA_OK)
        return s;
    if (!lse_part)
        return fail(DFA_ERR_INVALID_ARG, "lse_part is NULL");
    if ((s = check_ws(ws, ws_bytes, kStatusBytes)) != DFA_OK)
        return s;
    Layout lay;
    lay.qmaps.push_back(pair->q);
    lay.kmaps.push_back(pair->kv);
    lay.chunk_q = Lq;
    lay.chunk_k = Lk;
    return run_fwd(*desc, lay, q, k, v, o_part, lse_part, 1, ws, (cudaStream_t)stream);
}

dfa_status dfa_attn_bwd(const dfa_attn_desc* desc, const void* q, const void* k, const void* v,
                        const void* o, const void* dout, const float* lse, void* dq, void* dk,
                        void* dv, void* ws, size_t ws_bytes, void* stream)
{
    dfa_status s = check_desc(desc, true);
    if (s != DFA_OK)
        return s;
    if ((s = check_ptrs({q, k, v, o, dout, dq, dk, dv})) != DFA_OK)
        return s;
    if (!lse)
        return fail(DFA_ERR_INVALID_ARG, "lse is NULL");
    if ((s = check_ws(ws, ws_bytes, bwd_ws_bytes(*desc))) != DFA_OK)
        return s;
    cudaStream_t st = (cudaStream_t)stream;
    const int64_t rows = (int64_t)desc->B * desc->Hq * desc->N;
    float* dq_acc = reinterpret_cast<float*>((char*)ws + kStatusBytes);
    char* aug_lse = (char*)ws + kStatusBytes + align256((size_t)rows * desc->d * 4);
    char* aug_delta = aug_lse + align256((size_t)rows * kAugRowBytes);
    const int sms = num_sms();
    cudaError_t e = launch_bwd_preprocess(rows, desc->d, o, dout, nullptr, lse, desc->scale,
                                          aug_lse, aug_delta, dq_acc, sms, st);
    if (e != cudaSuccess)
        return cuda_fail(e, "backward preprocess launch");
    const bool blocked = bwd_blocked(desc->N, desc->Hq / desc->Hkv);
    const int64_t kv_elems = (int64_t)desc->B * desc->Hkv * desc->N * desc->d;
    float* dk_acc = nullptr;
    float* dv_acc = nullptr;
    if (blocked) {
        dk_acc = reinterpret_cast<float*>(aug_delta + align256((size_t)rows * kAugRowBytes));
        dv_acc = reinterpret_cast<float*>((char*)dk_acc + align256((size_t)kv_elems * 4));
        e = cudaMemsetAsync(dk_acc, 0, (size_t)kv_elems * 4, st);
        if (e == cudaSuccess)
            e = cudaMemsetAsync(dv_acc, 0, (size_t)kv_elems * 4, st);
        if (e != cudaSuccess)
            return cuda_fail(e, "dK/dV accumulator clear");
    }
    s = run_bwd_main(*desc, whole_layout(*desc), q, k, v, dout, aug_lse, aug_delta, dq_acc,
                     blocked ? (void*)dk_acc : dk, blocked ? (void*)dv_acc : dv, blocked ? 1 : 0,
                     ws, st);
    if (s != DFA_OK)
        return s;
    e = launch_f32_to_bf16(rows * desc->d, dq_acc, dq, sms, st);
    if (e == cudaSuccess && blocked)
        e = launch_f32_to_bf16(kv_elems, dk_acc, dk, sms, st);
    if (e == cudaSuccess && blocked)
        e = launch_f32_to_bf16(kv_elems, dv_acc, dv, sms, st);
    if (e != cudaSuccess)
        return cuda_fail(e, "dQ/dK/dV conversion launch");
    return DFA_OK;
}

dfa_status dfa_chunk_bwd(const dfa_attn_desc* desc, const dfa_chunk_pair* pair, int64_t Lq,
                         int64_t Lk, const void* q, const void* k, const void* v, const void* o,
                         const void* dout, const float* lse, const float* delta, float* dq_acc,
                         float* dk_acc, float* dv_acc, void* ws, size_t ws_bytes, void* stream)
{
    dfa_status s = check_desc(desc, false);
    if (s != DFA_OK)
        return s;
    if (!pair)
        return fail(DFA_ERR_INVALID_ARG, "pair is NULL");
    if (Lq < 1 || Lk < 1 || Lq >= INT32_MAX / 2 || Lk >= INT32_MAX / 2)
        return fail(DFA_ERR_INVALID_ARG, "chunk lengths must be in [1, 2^30)");
    if ((s = check_map(pair->q, Lq, "pair.q")) != DFA_OK)
        return s;
    if ((s = check_map(pair->kv, Lk, "pair.kv")) != DFA_OK)
        return s;
    if ((s = check_ptrs({q, k, v, dout, dq_acc, dk_acc, dv_acc})) != DFA_OK)
        return s;
    if (!lse)
        return fail(DFA_ERR_INVALID_ARG, "lse is NULL");
    const size_t rows = (size_t)desc->B * desc->Hq * (size_t)Lq;
    const size_t need = kStatusBytes + 2 * align256(rows * kAugRowBytes);
    if ((s = check_ws(ws, ws_bytes, need)) != DFA_OK)
        return s;
    cudaStream_t st = (cudaStream_t)stream;
    if (!delta && (s = check_ptrs({o})) != DFA_OK)
        return s;
    char* aug_lse = (char*)ws + kStatusBytes;
    char* aug_delta = aug_lse + align256(rows * kAugRowBytes);
    cudaError_t e = launch_bwd_preprocess((int64_t)rows, desc->d, delta ? nullptr : o, dout, delta,
                                          lse, desc->scale, aug_lse, aug_delta, nullptr,
                                          num_sms(), st);
    if (e != cudaSuccess)
        return cuda_fail(e, "backward preprocess launch");
    Layout lay;
    lay.qmaps.push_back(pair->q);
    lay.kmaps.push_back(pair->kv);
    lay.chunk_q = Lq;
    lay.chunk_k = Lk;
    return run_bwd_main(*desc, lay, q, k, v, dout, aug_lse, aug_delta, dq_acc, dk_acc, dv_acc, 1,
                        ws, st);
}

dfa_status dfa_lse_merge(int64_t rows, int32_t d, int32_t k, const float* o_parts,
                         const float* lse_parts, void* o_out, float* lse_out, int32_t out_fp32,
                         int32_t accumulate, void* stream)
{
    if (rows < 0)
        return fail(DFA_ERR_INVALID_ARG, "rows < 0");
    if (d != 64 && d != 128)
        return fail(DFA_ERR_UNSUPPORTED, "head dimension %d not supported", d);
    if (k < 0 || (k == 0 && !accumulate))
        return fail(DFA_ERR_INVALID_ARG, "need k >= 1 partials (or k = 0 with accumulate)");
    if (accumulate && !out_fp32)
        return fail(DFA_ERR_INVALID_ARG, "accumulate needs an fp32 output");
    if (!o_out || !lse_out || (k > 0 && (!o_parts || !lse_parts)))
        return fail(DFA_ERR_INVALID_ARG, "NULL pointer");
    if (!aligned16(o_out) || (k > 0 && !aligned16(o_parts)))
        return fail(DFA_ERR_UNSUPPORTED, "O pointers must be 16-byte aligned");
    if (rows == 0)
        return DFA_OK;
    cudaError_t e = launch_lse_merge(rows, d, k, o_parts, lse_parts, o_out, lse_out, out_fp32,
                                     accumulate, num_sms(), (cudaStream_t)stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "merge launch");
    return DFA_OK;
}

dfa_status dfa_permute(const dfa_attn_desc* desc, int32_t inverse, const void* in, void* out,
                       int32_t elem_bytes, int64_t row_elems, int64_t heads, void* stream)
{
    dfa_status s = check_desc(desc, true);
    if (s != DFA_OK)
        return s;
    if (!in || !out)
        return fail(DFA_ERR_INVALID_ARG, "NULL pointer");
    if (elem_bytes != 2 && elem_bytes != 4)
        return fail(DFA_ERR_INVALID_ARG, "elem_bytes must be 2 or 4");
    if (row_elems < 1 || heads < 1 || (row_elems * elem_bytes) % 4 != 0)
        return fail(DFA_ERR_INVALID_ARG, "row bytes must be a positive multiple of 4");
    const int64_t row_bytes = row_elems * elem_bytes;
    const int64_t bytes = heads * desc->N * row_bytes;
    const char* a = (const char*)in;
    const char* b = (const char*)out;
    if (a < b + bytes && b < a + bytes)
        return fail(DFA_ERR_INVALID_ARG, "in and out overlap");
    PermuteParams pp;
    memset(&pp, 0, sizeof pp);
    pp.heads = heads;
    pp.N = (int32_t)desc->N;
    pp.P = desc->P;
    pp.n = (int32_t)(desc->N / desc->P);
    pp.inverse = inverse ? 1 : 0;
    for (int p = 0; p < desc->P; ++p)
        pp.map[p] = to_dev(partition_map(*desc, p));
    const bool v16 = row_bytes % 16 == 0 && aligned16(in) && aligned16(out);
    const int vb = v16 ? 16 : 4;
    pp.row_vecs = (int32_t)(row_bytes / vb);
    cudaError_t e = launch_permute(pp, in, out, vb, num_sms(), (cudaStream_t)stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "permute launch");
    return DFA_OK;
}

dfa_status dfa_permute_rope(const dfa_attn_desc* desc, int32_t inverse, const void* in,
                            void* out, int64_t heads, float theta_base, void* stream)
{
    dfa_status s = check_desc(desc, true);
    if (s != DFA_OK)
        return s;
    if (!in || !out)
        return fail(DFA_ERR_INVALID_ARG, "NULL pointer");
    if (!aligned16(in) || !aligned16(out))
        return fail(DFA_ERR_UNSUPPORTED, "tensor pointers must be 16-byte aligned");
    if (heads < 1 || heads > (1 << 24))
        return fail(DFA_ERR_INVALID_ARG, "heads must be in [1, 2^24]");
    if (!(theta_base > 1.f) || !std::isfinite(theta_base))
        return fail(DFA_ERR_INVALID_ARG, "theta_base must be finite and > 1");
    const int64_t bytes = heads * desc->N * (int64_t)desc->d * 2;
    const char* a = (const char*)in;
    const char* b = (const char*)out;
    if (a < b + bytes && b < a + bytes)
        return fail(DFA_ERR_INVALID_ARG, "in and out overlap");
    RopeParams rp;
    memset(&rp, 0, sizeof rp);
    PermuteParams& pp = rp.perm;
    pp.heads = heads;
    pp.N = (int32_t)desc->N;
    pp.P = desc->P;
    pp.n = (int32_t)(desc->N / desc->P);
    pp.inverse = inverse ? 1 : 0;
    pp.row_vecs = desc->d / 8;
    for (int p = 0; p < desc->P; ++p)
        pp.map[p] = to_dev(partition_map(*desc, p));
    rp.d = desc->d;
    for (int t = 0; t < desc->d / 2; ++t)
        rp.theta[t] = std::pow((double)theta_base, -2.0 * t / desc->d);
    cudaError_t e = launch_permute_rope(rp, in, out, num_sms(), (cudaStream_t)stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "permute with rotary embedding launch");
    return DFA_OK;
}

size_t dfa_decode_workspace_size(const dfa_attn_desc* desc, int32_t T, int64_t L,
                                 int32_t split_len)
{
    if (check_desc(desc, false) != DFA_OK || T < 1 || L < 1 || split_len < 64 ||
        split_len % 64 != 0)
        return 0;
    const size_t splits = (size_t)((L + split_len - 1) / split_len);
    const size_t rows = (size_t)desc->B * desc->Hq * (size_t)T;
    return kStatusBytes + align256(splits * rows * desc->d * 4) + align256(splits * rows * 4);
}

dfa_status dfa_decode(const dfa_attn_desc* desc, int32_t T, int64_t L, int64_t q_pos0,
                      const void* q, const void* k, const void* v, void* o, float* lse,
                      int32_t split_len, void* ws, size_t ws_bytes, void* stream)
{
    dfa_status s = check_desc(desc, false);
    if (s != DFA_OK)
        return s;
    if (T < 1 || L < 1 || L >= INT32_MAX || q_pos0 < 0)
        return fail(DFA_ERR_INVALID_ARG, "need T >= 1, 1 <= L < 2^31, q_pos0 >= 0");
    if (desc->ndocs != 0)
        return fail(DFA_ERR_UNSUPPORTED, "dfa_decode takes no document bounds");
    if (split_len < 64 || split_len % 64 != 0)
        return fail(DFA_ERR_INVALID_ARG, "split_len must be a positive multiple of 64");
    const int G = desc->Hq / desc->Hkv;
    if ((int64_t)G * T > decode_max_rows())
        return fail(DFA_ERR_UNSUPPORTED, "decode handles at most %d query rows per key/value "
                    "head (Hq/Hkv * T)", decode_max_rows());
    if ((s = check_ptrs({q, k, v, o})) != DFA_OK)
        return s;
    if (!lse)
        return fail(DFA_ERR_INVALID_ARG, "lse is NULL");
    const size_t need = dfa_decode_workspace_size(desc, T, L, split_len);
    if ((s = check_ws(ws, ws_bytes, need)) != DFA_OK)
        return s;
    const int splits = (int)((L + split_len - 1) / split_len);
    if ((int64_t)splits > 65535 * 1024)
        return fail(DFA_ERR_UNSUPPORTED, "too many splits");
    const size_t rows = (size_t)desc->B * desc->Hq * (size_t)T;
    DecodeParams p;
    memset(&p, 0, sizeof p);
    p.B = desc->B;
    p.Hq = desc->Hq;
    p.Hkv = desc->Hkv;
    p.G = G;
    p.T = T;
    p.L = (int32_t)L;
    p.split_len = split_len;
    p.causal = desc->causal;
    p.q_pos0 = q_pos0;
    p.scale_log2 = desc->scale * 1.4426950408889634f;
    p.q = q;
    p.k = k;
    p.v = v;
    p.o_part = reinterpret_cast<float*>((char*)ws + kStatusBytes);
    p.lse_part = reinterpret_cast<float*>((char*)ws + kStatusBytes +
                                          align256((size_t)splits * rows * desc->d * 4));
    cudaStream_t st = (cudaStream_t)stream;
    if ((int64_t)desc->B * desc->Hkv > 65535)
        return fail(DFA_ERR_UNSUPPORTED, "B * Hkv must be at most 65535");
    cudaError_t e = launch_decode_split(desc->d, p, splits, st);
    if (e != cudaSuccess)
        return cuda_fail(e, "decode launch");
    e = launch_lse_merge((int64_t)rows, desc->d, splits, p.o_part, p.lse_part, o, lse,
                         desc->o_fp32, 0, num_sms(), st);
    if (e != cudaSuccess)
        return cuda_fail(e, "merge launch");
    return DFA_OK;
}

dfa_status dfa_make_schedule(const dfa_attn_desc* desc, int32_t tile_m, int32_t tile_n,
                             dfa_schedule* out)
{
    dfa_status s = check_desc(desc, true);
    if (s != DFA_OK)
        return s;
    if (!out)
        return fail(DFA_ERR_INVALID_ARG, "schedule output is NULL");
    if (tile_m < 1 || tile_n < 1)
        return fail(DFA_ERR_INVALID_ARG, "tile sizes must be positive");
    if (out->capacity < 0)
        return fail(DFA_ERR_INVALID_ARG, "item capacity must be >= 0");
    const int P = desc->P;
    const int32_t n = (int32_t)(desc->N / P);
    const int32_t nqt = (n + tile_m - 1) / tile_m, nkt = (n + tile_n - 1) / tile_n;
    std::vector<DevMap> maps(P);
    for (int p = 0; p < P; ++p)
        maps[p] = to_dev(partition_map(*desc, p));
    // Key tiles [0, vis) of the kv chunk are seen by query tile qt, tiles
    // [0, full) by every row of it (positions increase along each chunk, so
    // both sets are prefixes).
    auto tile_prefixes = [&](const DevMap& qm, const DevMap& km, int32_t qt, int32_t& vis,
                             int32_t& full) {
        if (!desc->causal) {
            vis = full = nkt;
            return;
        }
        const int32_t q0 = qt * tile_m, q1 = std::min(n, q0 + tile_m) - 1;
        const int32_t cmax = map_count_le(km, map_pos(qm, q1));
        const int32_t cmin = map_count_le(km, map_pos(qm, q0));
        vis = (cmax + tile_n - 1) / tile_n;
        full = (cmin == n) ? nkt : cmin / tile_n;
    };
    // pass 1: loads, tile counts and the number of items
    std::vector<int64_t> tokens((size_t)P * P), counts((size_t)P * P * 3), nitems((size_t)P * P);
    int64_t total = 0, items_total = 0;
    for (int p = 0; p < P; ++p) {
        for (int st = 0; st < P; ++st) {
            const int w = ((p - st) % P + P) % P;
            const DevMap& qm = maps[p];
            const DevMap& km = maps[w];
            int64_t pairs = 0;
            if (desc->causal) {
                for (int32_t m = 0; m < n; ++m)
                    pairs += map_count_le(km, map_pos(qm, m));
            } else {
                pairs = (int64_t)n * n;
            }
            const size_t ps = (size_t)p * P + st;
            tokens[ps] = pairs;
            total += pairs;
            int64_t cnt[3] = {0, 0, 0}, ni = 0;
            for (int32_t qt = 0; qt < nqt; ++qt) {
                int32_t vis, full;
                tile_prefixes(qm, km, qt, vis, full);
                cnt[DFA_TILE_SKIP] += nkt - vis;
                cnt[DFA_TILE_FULL] += full;
                cnt[DFA_TILE_PARTIAL] += vis - full;
                ni += (full > 0) + (vis > full) + (nkt > vis);
            }
            for (int c = 0; c < 3; ++c)
                counts[ps * 3 + c] = cnt[c];
            nitems[ps] = ni;
            items_total += ni;
        }
    }
    out->n_items = items_total;
    const bool write_items = out->items != nullptr && out->capacity > 0;
    if (write_items && out->capacity < items_total)
        return fail(DFA_ERR_INVALID_ARG, "item buffer too small: %lld < %lld",
                    (long long)out->capacity, (long long)items_total);
    // pass 2: outputs
    int64_t first = 0;
    for (int p = 0; p < P; ++p) {
        for (int st = 0; st < P; ++st) {
            const int w = ((p - st) % P + P) % P;
            const size_t ps = (size_t)p * P + st;
            if (out->pair_tokens)
                out->pair_tokens[ps] = tokens[ps];
            if (out->tile_counts)
                for (int c = 0; c < 3; ++c)
                    out->tile_counts[ps * 3 + c] = counts[ps * 3 + c];
            if (out->pairs) {
                dfa_sched_pair& pr = out->pairs[ps];
                pr.worker = p;
                pr.step = st;
                pr.kv_worker = w;
                pr.reserved = 0;
                pr.tokens = tokens[ps];
                pr.first_item = first;
                pr.n_items = nitems[ps];
            }
            if (write_items) {
                int64_t k = first;
                for (int32_t qt = 0; qt < nqt; ++qt) {
                    int32_t vis, full;
                    tile_prefixes(maps[p], maps[w], qt, vis, full);
                    const int32_t rb[3][3] = {{0, full, DFA_TILE_FULL},
                                              {full, vis, DFA_TILE_PARTIAL},
                                              {vis, nkt, DFA_TILE_SKIP}};
                    for (const auto& r : rb) {
                        if (r[1] <= r[0])
                            continue;
                        dfa_sched_item& it = out->items[k++];
                        it.worker = p;
                        it.step = st;
                        it.q_tile = qt;
                        it.kv_begin = r[0];
                        it.kv_end = r[1];
                        it.mask_class = r[2];
                    }
                }
            }
            first += nitems[ps];
        }
    }
    out->total_pairs = total;
    int64_t nonempty = 0, lockstep = 0;
    for (int st = 0; st < P; ++st) {
        int64_t mx = 0;
        for (int p = 0; p < P; ++p) {
            const int64_t v = tokens[(size_t)p * P + st];
            if (v > 0)
                ++nonempty;
            mx = std::max(mx, v);
        }
        lockstep += mx;
    }
    out->eta_slots = (double)nonempty / ((double)P * P);
    out->eta_flops = lockstep > 0 ? (double)total / ((double)P * lockstep) : 1.0;
    return DFA_OK;
}

dfa_status dfa_stream_status(void* ws, void* stream)
{
    if (!ws)
        return fail(DFA_ERR_WORKSPACE, "workspace is NULL");
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "stream synchronize");
    DevStatus h{};
    e = cudaMemcpy(&h, ws, sizeof h, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess)
        return cuda_fail(e, "status read");
    if (h.code != 0) {
        DevStatus z{};
        cudaMemcpy(ws, &z, sizeof z, cudaMemcpyHostToDevice);
        return fail((dfa_status)h.code, "device status %d at wait site %d (block %d)", h.code,
                    h.where, h.detail);
    }
    return DFA_OK;
}

dfa_status dfa_selftest_timeout(void* ws, int64_t timeout_us, void* stream)
{
    if (!ws || ((uintptr_t)ws & 255u))
        return fail(DFA_ERR_WORKSPACE, "workspace is NULL or misaligned");
    if (timeout_us < 1 || timeout_us > 10000000)
        return fail(DFA_ERR_INVALID_ARG, "timeout_us must be in [1, 1e7]");
    cudaError_t e = launch_selftest_timeout(status_word(ws), (uint64_t)timeout_us * 1000ull,
                                            (cudaStream_t)stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "self-test launch");
    return DFA_OK;
}

}  // extern "C"
