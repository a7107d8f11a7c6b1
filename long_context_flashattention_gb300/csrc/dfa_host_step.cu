// dfa_host_step.cu -- the host-streaming executor: one attention training
// step (permute, forward, recomputation backward, permute back) whose tensors
// live in host memory, cut into groups of whole key/value heads so that the
// copies of neighbouring groups overlap a group's compute.
//
// Host code only.  Per group g (slot s = g % 2 of the double-buffered
// staging):
//   h2d stream:      [wait in_free[s]]  upload q, k, v, dO of g  -> up[s]
//   compute stream s: wait up[s]; permute in -> in_free[s]; [wait down[s]]
//                    forward; [wait bwd]; backward -> bwd; permute out into
//                    out staging[s] -> done
//   d2h stream:      wait done; download o, lse, dq, dk, dv of g -> down[s]
// (compute stream 0 is the caller's, stream 1 the call's own when the copies
// have streams of their own; otherwise both are the caller's).
// in_free[s] lets the upload of g+2 reuse the input slot once g's inputs are
// consumed; down[s] keeps the compute of g+2 from overwriting the output
// slot before g's download has read it.  When the partition's storage order
// is natural order (P = 1, contiguous, or stripes as long as a chunk) the
// permutes are skipped: the compute reads the input slot and writes the
// output slot directly, and in_free[s] is recorded after the backward.
#include <cstdint>
#include <cstring>
#include <vector>

#include <cuda_runtime.h>

#include "../../include/dfa.h"

namespace dfa {
dfa_status set_error(dfa_status s, const char* fmt, ...);
}

namespace {

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// The library's group size: the fewest key/value heads per group whose
// backward still has at least kUnitsPerGroup key-tile units (about 16 per SM
// of a GB300, so that a group's launches are not dominated by their last,
// partly idle wave), and at least two groups where B*Hkv allows, so that
// copies overlap compute inside a step.  Measured end to end at the 32K
// Llama-7B shape (32 heads, 3 steps per call): 8 groups of 4 heads 870
// TFLOP/s, 4 groups 954, 2 groups 1016, 1 group 980.
constexpr int64_t kUnitsPerGroup = 16 * 152;

int auto_group(const dfa_attn_desc& d)
{
    const int64_t tiles = (d.N + 127) / 128;
    int best = d.Hkv;
    for (int g = d.Hkv; g >= 1; --g) {
        if (d.Hkv % g != 0)
            continue;
        const bool big = (int64_t)g * tiles >= kUnitsPerGroup;
        const bool several = (int64_t)d.B * (d.Hkv / g) >= 2 || (d.B == 1 && d.Hkv == 1);
        if (big && several)
            best = g;
    }
    if ((int64_t)d.B * (d.Hkv / best) < 2) {
        // too small a problem for the size rule: at least two groups
        for (int g = d.Hkv / 2; g >= 1; --g)
            if (d.Hkv % g == 0) {
                best = g;
                break;
            }
    }
    return best;
}

dfa_attn_desc group_desc(const dfa_attn_desc& d, int gk)
{
    dfa_attn_desc g = d;
    g.B = 1;
    g.Hkv = gk;
    g.Hq = gk * (d.Hq / d.Hkv);
    return g;
}

// Natural order is the storage order: every worker's rows are one run of
// positions starting at p n.
bool identity_order(const dfa_attn_desc& d)
{
    const int64_t n = d.N / d.P;
    for (int p = 0; p < d.P; ++p) {
        dfa_pos_map m;
        if (dfa_partition_map(&d, p, &m) != DFA_OK)
            return false;
        if (m.nseg != 1 || m.base[0] != (int64_t)p * n ||
            !(m.len[0] <= m.blk || m.blk_stride == m.blk))
            return false;
    }
    return true;
}

// Byte sizes of one group's tensors and the workspace layout built on them.
struct Plan {
    int gk = 0, groups = 0;
    bool ident = false;
    dfa_attn_desc gd{};
    size_t qb = 0, kb = 0, lb = 0;      // one group's q (= o, dq, dO), k (= v, dk, dv), lse
    size_t bwd_ws = 0;                   // the group backward's workspace (status word first)
    size_t in_set = 0, out_set = 0;      // one input set (q k v dO), one output set
    size_t off_in[2] = {0, 0}, off_out[2] = {0, 0}, off_pin[2] = {0, 0}, off_pout[2] = {0, 0};
    size_t total = 0;
};

dfa_status make_plan(const dfa_attn_desc* desc, int32_t kv_heads_per_group, Plan& pl)
{
    if (dfa_workspace_size(desc, DFA_OP_BWD) == 0)  // validates desc, sets the error text
        return DFA_ERR_INVALID_ARG;
    if (desc->o_fp32 != 0)
        return dfa::set_error(DFA_ERR_UNSUPPORTED, "dfa_attn_step_host: O is bf16 here "
                              "(desc->o_fp32 must be 0)");
    if (kv_heads_per_group < 0 || (kv_heads_per_group > 0 && desc->Hkv % kv_heads_per_group))
        return dfa::set_error(DFA_ERR_INVALID_ARG, "dfa_attn_step_host: kv_heads_per_group "
                              "(%d) must be 0 or divide Hkv (%d)", kv_heads_per_group,
                              desc->Hkv);
    pl.gk = kv_heads_per_group ? kv_heads_per_group : auto_group(*desc);
    pl.groups = desc->B * (desc->Hkv / pl.gk);
    pl.gd = group_desc(*desc, pl.gk);
    pl.ident = identity_order(*desc);
    const size_t rows_q = (size_t)pl.gd.Hq * desc->N, rows_k = (size_t)pl.gk * desc->N;
    pl.qb = rows_q * desc->d * 2;
    pl.kb = rows_k * desc->d * 2;
    pl.lb = rows_q * 4;
    pl.bwd_ws = dfa_workspace_size(&pl.gd, DFA_OP_BWD);
    if (pl.bwd_ws == 0)
        return DFA_ERR_INVALID_ARG;
    pl.in_set = 2 * align256(pl.qb) + 2 * align256(pl.kb);
    pl.out_set = 2 * align256(pl.qb) + align256(pl.lb) + 2 * align256(pl.kb);
    size_t off = align256(pl.bwd_ws);
    for (int s = 0; s < 2; ++s) {
        pl.off_in[s] = off;
        off += pl.in_set;
    }
    for (int s = 0; s < 2; ++s) {
        pl.off_out[s] = off;
        off += pl.out_set;
    }
    for (int s = 0; s < 2; ++s) {
        pl.off_pin[s] = pl.off_pout[s] = off;
        if (!pl.ident) {  // the worker-major copies the kernels read and write
            pl.off_pin[s] = off;
            off += pl.in_set;
            pl.off_pout[s] = off;
            off += pl.out_set;
        }
    }
    pl.total = off;
    return DFA_OK;
}

// The five tensors of an input set (q, k, v, dO) or output set (o, lse, dq,
// dk, dv) at base.
struct InSet {
    char *q, *k, *v, *dout;
};
struct OutSet {
    char *o, *lse, *dq, *dk, *dv;
};

InSet in_set(char* base, const Plan& pl)
{
    InSet s;
    s.q = base;
    s.k = s.q + align256(pl.qb);
    s.v = s.k + align256(pl.kb);
    s.dout = s.v + align256(pl.kb);
    return s;
}

OutSet out_set(char* base, const Plan& pl)
{
    OutSet s;
    s.o = base;
    s.lse = s.o + align256(pl.qb);
    s.dq = s.lse + align256(pl.lb);
    s.dk = s.dq + align256(pl.qb);
    s.dv = s.dk + align256(pl.kb);
    return s;
}

struct Events {
    enum {
        kEntry, kUp0, kUp1, kInFree0, kInFree1, kDone, kDown0, kDown1, kTailUp, kBwd, kTail1,
        kCount
    };
    cudaEvent_t e[kCount] = {};
    ~Events()
    {
        for (cudaEvent_t x : e)
            if (x)
                cudaEventDestroy(x);
    }
    cudaError_t create()
    {
        for (cudaEvent_t& x : e) {
            cudaError_t r = cudaEventCreateWithFlags(&x, cudaEventDisableTiming);
            if (r != cudaSuccess)
                return r;
        }
        return cudaSuccess;
    }
};

dfa_status cuda_err(cudaError_t e, const char* what)
{
    return dfa::set_error(DFA_ERR_CUDA, "dfa_attn_step_host: %s: %s", what,
                          cudaGetErrorString(e));
}

}  // namespace

extern "C" size_t dfa_attn_step_host_workspace_size(const dfa_attn_desc* desc,
                                                    int32_t kv_heads_per_group)
{
    Plan pl;
    return make_plan(desc, kv_heads_per_group, pl) == DFA_OK ? pl.total : 0;
}

namespace {

// Host tensors of one step.
struct HostStep {
    const void *q, *k, *v, *dout;
    void *o, *dq, *dk, *dv;
    float* lse;
};

// One unit of streamed work: key/value heads [h0, h0 + gk) of batch entry b
// of step t, with their query heads.
struct Item {
    int32_t t, b, h0, gk;
};

// The (step, group) items of nsteps steps, in order: step-major, groups of
// pl.gk key/value heads inside a step, so the uploads of a step's first
// groups overlap the compute of the previous step's last groups.  Only the
// first upload and the last download of the whole call overlap nothing; with
// the library's own group size (ramp = true) the first and the last item are
// cut into a quarter and three quarters, so that those two copies move a
// quarter of a group.
std::vector<Item> make_items(const dfa_attn_desc& d, const Plan& pl, int32_t nsteps, bool ramp)
{
    std::vector<Item> it;
    const int per_b = d.Hkv / pl.gk;
    for (int32_t t = 0; t < nsteps; ++t)
        for (int g = 0; g < pl.groups; ++g)
            it.push_back({t, g / per_b, (g % per_b) * pl.gk, pl.gk});
    if (ramp && pl.gk >= 4) {
        const int32_t q = pl.gk / 4;
        Item f = it.front();
        it.front() = {f.t, f.b, f.h0, q};
        it.insert(it.begin() + 1, Item{f.t, f.b, f.h0 + q, f.gk - q});
        Item l = it.back();
        if (l.gk >= 4) {
            const int32_t ql = l.gk / 4;
            it.back() = {l.t, l.b, l.h0, l.gk - ql};
            it.push_back({l.t, l.b, l.h0 + l.gk - ql, ql});
        }
    }
    return it;
}

dfa_status run_steps(const dfa_attn_desc* desc, int32_t nsteps, const HostStep* hs,
                     int32_t kv_heads_per_group, void* ws, size_t ws_bytes, void* compute_stream,
                     void* h2d_stream, void* d2h_stream)
{
    Plan pl;
    dfa_status st = make_plan(desc, kv_heads_per_group, pl);
    if (st != DFA_OK)
        return st;
    if (nsteps < 1 || !hs)
        return dfa::set_error(DFA_ERR_INVALID_ARG, "dfa_attn_step_host: need nsteps >= 1");
    for (int32_t t = 0; t < nsteps; ++t) {
        const HostStep& h = hs[t];
        if (!h.q || !h.k || !h.v || !h.dout || !h.o || !h.lse || !h.dq || !h.dk || !h.dv)
            return dfa::set_error(DFA_ERR_INVALID_ARG,
                                  "dfa_attn_step_host: a host pointer of step %d is NULL", t);
    }
    if (!ws || ((uintptr_t)ws & 255u) || ws_bytes < pl.total)
        return dfa::set_error(DFA_ERR_WORKSPACE, "dfa_attn_step_host: workspace must be "
                              "256-byte aligned and hold %zu bytes", pl.total);
    const cudaStream_t cs = (cudaStream_t)compute_stream;
    const cudaStream_t up = h2d_stream ? (cudaStream_t)h2d_stream : cs;
    const cudaStream_t dn = d2h_stream ? (cudaStream_t)d2h_stream : cs;
    Events ev;
    cudaError_t e = ev.create();
    if (e != cudaSuccess)
        return cuda_err(e, "event creation");
    // the staging slots may still be read by earlier work on compute_stream
    e = cudaEventRecord(ev.e[Events::kEntry], cs);
    if (e == cudaSuccess && up != cs)
        e = cudaStreamWaitEvent(up, ev.e[Events::kEntry], 0);
    if (e == cudaSuccess && dn != cs)
        e = cudaStreamWaitEvent(dn, ev.e[Events::kEntry], 0);
    if (e != cudaSuccess)
        return cuda_err(e, "entry ordering");

    // Two compute streams when the copies run beside the compute: items of
    // slot 0 on compute_stream, items of slot 1 on a stream of the call's
    // own, so that one group's forward starts on the SMs that the previous
    // group's backward releases in its last wave.  Each slot has its own
    // staging and worker-major copies; the backwards share the workspace's
    // scratch and run one after another.
    struct OwnStream {
        cudaStream_t s = nullptr;
        ~OwnStream()
        {
            if (s)
                cudaStreamDestroy(s);
        }
    } own;
    cudaStream_t comp[2] = {cs, cs};
    if (up != cs || dn != cs) {
        e = cudaStreamCreateWithFlags(&own.s, cudaStreamNonBlocking);
        if (e == cudaSuccess)
            e = cudaStreamWaitEvent(own.s, ev.e[Events::kEntry], 0);
        if (e != cudaSuccess)
            return cuda_err(e, "second compute stream");
        comp[1] = own.s;
    }

    char* base = (char*)ws;
    const int r = desc->Hq / desc->Hkv;
    const int64_t d = desc->d;
    const std::vector<Item> work = make_items(*desc, pl, nsteps, kv_heads_per_group == 0);
    const int64_t items = (int64_t)work.size();
    // element offsets of an item's first query / key row in [B,H,N,d] tensors
    auto host_off_q = [&](const Item& w) {
        return ((int64_t)w.b * desc->Hq + (int64_t)w.h0 * r) * desc->N;
    };
    auto host_off_k = [&](const Item& w) {
        return ((int64_t)w.b * desc->Hkv + w.h0) * desc->N;
    };
    // bytes of an item's q (= o, dq, dO), k (= v, dk, dv) and lse
    auto q_bytes = [&](const Item& w) { return (size_t)w.gk * r * desc->N * d * 2; };
    auto k_bytes = [&](const Item& w) { return (size_t)w.gk * desc->N * d * 2; };
    auto l_bytes = [&](const Item& w) { return (size_t)w.gk * r * desc->N * 4; };
    auto upload = [&](int64_t i) -> cudaError_t {
        const int s = (int)(i % 2);
        const Item& w = work[i];
        const HostStep& h = hs[w.t];
        const InSet in = in_set(base + pl.off_in[s], pl);
        const int64_t oq = host_off_q(w) * d * 2, ok = host_off_k(w) * d * 2;
        const size_t qb = q_bytes(w), kb = k_bytes(w);
        cudaError_t x = cudaSuccess;
        if (i >= 2)
            x = cudaStreamWaitEvent(up, ev.e[Events::kInFree0 + s], 0);
        if (x == cudaSuccess)
            x = cudaMemcpyAsync(in.q, (const char*)h.q + oq, qb, cudaMemcpyHostToDevice, up);
        if (x == cudaSuccess)
            x = cudaMemcpyAsync(in.k, (const char*)h.k + ok, kb, cudaMemcpyHostToDevice, up);
        if (x == cudaSuccess)
            x = cudaMemcpyAsync(in.v, (const char*)h.v + ok, kb, cudaMemcpyHostToDevice, up);
        if (x == cudaSuccess)
            x = cudaMemcpyAsync(in.dout, (const char*)h.dout + oq, qb, cudaMemcpyHostToDevice,
                                up);
        if (x == cudaSuccess)
            x = cudaEventRecord(ev.e[Events::kUp0 + s], up);
        return x;
    };
    auto download = [&](int64_t i) -> cudaError_t {
        const int s = (int)(i % 2);
        const Item& w = work[i];
        const HostStep& h = hs[w.t];
        const OutSet out = out_set(base + pl.off_out[s], pl);
        const int64_t oq = host_off_q(w) * d * 2, ok = host_off_k(w) * d * 2;
        const int64_t ol = host_off_q(w) * 4;
        const size_t qb = q_bytes(w), kb = k_bytes(w), lb = l_bytes(w);
        cudaError_t x = cudaStreamWaitEvent(dn, ev.e[Events::kDone], 0);
        if (x == cudaSuccess)
            x = cudaMemcpyAsync((char*)h.o + oq, out.o, qb, cudaMemcpyDeviceToHost, dn);
        if (x == cudaSuccess)
            x = cudaMemcpyAsync((char*)h.lse + ol, out.lse, lb, cudaMemcpyDeviceToHost, dn);
        if (x == cudaSuccess)
            x = cudaMemcpyAsync((char*)h.dq + oq, out.dq, qb, cudaMemcpyDeviceToHost, dn);
        if (x == cudaSuccess)
            x = cudaMemcpyAsync((char*)h.dk + ok, out.dk, kb, cudaMemcpyDeviceToHost, dn);
        if (x == cudaSuccess)
            x = cudaMemcpyAsync((char*)h.dv + ok, out.dv, kb, cudaMemcpyDeviceToHost, dn);
        if (x == cudaSuccess)
            x = cudaEventRecord(ev.e[Events::kDown0 + s], dn);
        return x;
    };
    auto compute = [&](int64_t i) -> dfa_status {
        const int s = (int)(i % 2);
        const cudaStream_t c = comp[s];
        const InSet in = in_set(base + pl.off_in[s], pl);
        const OutSet out = out_set(base + pl.off_out[s], pl);
        const InSet pin = pl.ident ? in : in_set(base + pl.off_pin[s], pl);
        const OutSet pout = pl.ident ? out : out_set(base + pl.off_pout[s], pl);
        const dfa_attn_desc item_desc = group_desc(*desc, work[i].gk);
        const dfa_attn_desc* gd = &item_desc;
        const int64_t heads_q = item_desc.Hq, heads_k = item_desc.Hkv;
        cudaError_t x = cudaStreamWaitEvent(c, ev.e[Events::kUp0 + s], 0);
        if (x != cudaSuccess)
            return cuda_err(x, "stream wait");
        dfa_status t = DFA_OK;
        if (!pl.ident) {
            t = dfa_permute(gd, 0, in.q, pin.q, 2, d, heads_q, c);
            if (t == DFA_OK)
                t = dfa_permute(gd, 0, in.k, pin.k, 2, d, heads_k, c);
            if (t == DFA_OK)
                t = dfa_permute(gd, 0, in.v, pin.v, 2, d, heads_k, c);
            if (t == DFA_OK)
                t = dfa_permute(gd, 0, in.dout, pin.dout, 2, d, heads_q, c);
            if (t != DFA_OK)
                return t;
            if ((x = cudaEventRecord(ev.e[Events::kInFree0 + s], c)) != cudaSuccess)
                return cuda_err(x, "event record");
        }
        // the output slot was last read by the download of item i - 2
        if (pl.ident && i >= 2 && dn != c &&
            (x = cudaStreamWaitEvent(c, ev.e[Events::kDown0 + s], 0)) != cudaSuccess)
            return cuda_err(x, "stream wait");
        t = dfa_attn_fwd(gd, pin.q, pin.k, pin.v, pout.o, (float*)pout.lse, ws, 256, c);
        if (t != DFA_OK)
            return t;
        // the backwards share one workspace: item i's after item i - 1's
        if (i >= 1 && comp[1] != comp[0] &&
            (x = cudaStreamWaitEvent(c, ev.e[Events::kBwd], 0)) != cudaSuccess)
            return cuda_err(x, "stream wait");
        t = dfa_attn_bwd(gd, pin.q, pin.k, pin.v, pout.o, pin.dout, (const float*)pout.lse,
                         pout.dq, pout.dk, pout.dv, ws, pl.bwd_ws, c);
        if (t != DFA_OK)
            return t;
        if ((x = cudaEventRecord(ev.e[Events::kBwd], c)) != cudaSuccess)
            return cuda_err(x, "event record");
        if (pl.ident) {
            if ((x = cudaEventRecord(ev.e[Events::kInFree0 + s], c)) != cudaSuccess)
                return cuda_err(x, "event record");
        } else {
            if (i >= 2 && dn != c &&
                (x = cudaStreamWaitEvent(c, ev.e[Events::kDown0 + s], 0)) != cudaSuccess)
                return cuda_err(x, "stream wait");
            t = dfa_permute(gd, 1, pout.o, out.o, 2, d, heads_q, c);
            if (t == DFA_OK)
                t = dfa_permute(gd, 1, pout.lse, out.lse, 4, 1, heads_q, c);
            if (t == DFA_OK)
                t = dfa_permute(gd, 1, pout.dq, out.dq, 2, d, heads_q, c);
            if (t == DFA_OK)
                t = dfa_permute(gd, 1, pout.dk, out.dk, 2, d, heads_k, c);
            if (t == DFA_OK)
                t = dfa_permute(gd, 1, pout.dv, out.dv, 2, d, heads_k, c);
            if (t != DFA_OK)
                return t;
        }
        if ((x = cudaEventRecord(ev.e[Events::kDone], c)) != cudaSuccess)
            return cuda_err(x, "event record");
        return DFA_OK;
    };

    // Issue order: the next item's upload goes into its queue before this
    // item's compute, so the copy engine never waits on the host.
    e = upload(0);
    if (e != cudaSuccess)
        st = cuda_err(e, "upload");
    for (int64_t i = 0; i < items && st == DFA_OK; ++i) {
        if (i + 1 < items && (e = upload(i + 1)) != cudaSuccess) {
            st = cuda_err(e, "upload");
            break;
        }
        if ((st = compute(i)) != DFA_OK)
            break;
        if ((e = download(i)) != cudaSuccess)
            st = cuda_err(e, "download");
    }
    // Join: everything queued on the copy streams and the second compute
    // stream is ordered before later work on compute_stream, on success and
    // on error alike.
    cudaError_t j = cudaSuccess;
    if (comp[1] != cs) {
        j = cudaEventRecord(ev.e[Events::kTail1], comp[1]);
        if (j == cudaSuccess)
            j = cudaStreamWaitEvent(cs, ev.e[Events::kTail1], 0);
    }
    if (j == cudaSuccess && up != cs) {
        j = cudaEventRecord(ev.e[Events::kTailUp], up);
        if (j == cudaSuccess)
            j = cudaStreamWaitEvent(cs, ev.e[Events::kTailUp], 0);
    }
    if (j == cudaSuccess && dn != cs) {
        j = cudaEventRecord(ev.e[Events::kDone], dn);
        if (j == cudaSuccess)
            j = cudaStreamWaitEvent(cs, ev.e[Events::kDone], 0);
    }
    if (st == DFA_OK && j != cudaSuccess)
        st = cuda_err(j, "join");
    return st;
}

}  // namespace

extern "C" dfa_status dfa_attn_step_host(const dfa_attn_desc* desc, const void* h_q,
                                         const void* h_k, const void* h_v, const void* h_dout,
                                         void* h_o, float* h_lse, void* h_dq, void* h_dk,
                                         void* h_dv, int32_t kv_heads_per_group, void* ws,
                                         size_t ws_bytes, void* compute_stream,
                                         void* h2d_stream, void* d2h_stream)
{
    const HostStep h{h_q, h_k, h_v, h_dout, h_o, h_dq, h_dk, h_dv, h_lse};
    return run_steps(desc, 1, &h, kv_heads_per_group, ws, ws_bytes, compute_stream, h2d_stream,
                     d2h_stream);
}

extern "C" dfa_status dfa_attn_steps_host(const dfa_attn_desc* desc, int32_t nsteps,
                                          const dfa_host_step* steps, int32_t kv_heads_per_group,
                                          void* ws, size_t ws_bytes, void* compute_stream,
                                          void* h2d_stream, void* d2h_stream)
{
    if (nsteps < 1 || !steps)
        return dfa::set_error(DFA_ERR_INVALID_ARG, "dfa_attn_steps_host: need nsteps >= 1 and "
                              "a step array");
    // dfa_host_step and HostStep hold the same pointers; copy field by field
    constexpr int32_t kChunk = 64;
    HostStep hs[kChunk];
    if (nsteps > kChunk)
        return dfa::set_error(DFA_ERR_UNSUPPORTED, "dfa_attn_steps_host: at most %d steps per "
                              "call", kChunk);
    for (int32_t t = 0; t < nsteps; ++t)
        hs[t] = HostStep{steps[t].q, steps[t].k, steps[t].v, steps[t].dout, steps[t].o,
                         steps[t].dq, steps[t].dk, steps[t].dv, steps[t].lse};
    return run_steps(desc, nsteps, hs, kv_heads_per_group, ws, ws_bytes, compute_stream,
                     h2d_stream, d2h_stream);
}
