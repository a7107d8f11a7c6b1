// dfa_ring.cu -- the ring schedule of context-parallel attention, emulated on
// one GPU with its own workers' buffers (DistFlashAttn Guide, "Core
// Innovation" ring: each worker computes against the key/value chunk it holds
// while the next one arrives; Striped Attention Guide, "Workload Balance
// Theorem": at ring step s worker p holds the keys of worker (p - s) mod P).
//
// Host code only: every step is a dfa_chunk_fwd per worker followed by an
// in-place LSE merge into the worker's running (O, LSE), on the compute
// stream; the "send" of each worker's current K/V to its successor is a
// device-to-device copy on the copy stream into one of the successor's two
// receive slots, overlapping the step's compute.  Two slots per worker
// suffice: the slot written at step s was last read (as the current K/V, and
// as the source of the successor's copy) at step s - 1.
#include <cstdint>
#include <cstring>

#include <cuda_runtime.h>

#include "../../include/dfa.h"

namespace dfa {
dfa_status set_error(dfa_status s, const char* fmt, ...);
}

namespace {

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct EventPair {
    cudaEvent_t comp = nullptr, copy = nullptr;
    ~EventPair()
    {
        if (comp)
            cudaEventDestroy(comp);
        if (copy)
            cudaEventDestroy(copy);
    }
};

dfa_status cuda_err(cudaError_t e, const char* what)
{
    return dfa::set_error(DFA_ERR_CUDA, "dfa_ring_fwd: %s: %s", what, cudaGetErrorString(e));
}

}  // namespace

extern "C" dfa_status dfa_ring_fwd(const dfa_attn_desc* desc, const dfa_ring_worker* workers,
                                   void* ws, size_t ws_bytes, int32_t overlap,
                                   void* compute_stream, void* copy_stream)
{
    if (!desc || !workers)
        return dfa::set_error(DFA_ERR_INVALID_ARG, "dfa_ring_fwd: NULL desc or workers");
    const int P = desc->P;
    dfa_pos_map maps[64];
    if (P < 1 || P > 64)
        return dfa::set_error(DFA_ERR_INVALID_ARG, "dfa_ring_fwd: P must be in [1, 64]");
    for (int p = 0; p < P; ++p) {
        const dfa_status s = dfa_partition_map(desc, p, &maps[p]);  // also checks desc
        if (s != DFA_OK)
            return s;
    }
    const int64_t n = desc->N / P;
    const size_t rows = (size_t)desc->B * desc->Hq * (size_t)n;
    const size_t kv_bytes = (size_t)desc->B * desc->Hkv * (size_t)n * desc->d * 2;
    const size_t need = dfa_workspace_size(desc, DFA_OP_RING_FWD);
    if (!ws || ((uintptr_t)ws & 255u) || ws_bytes < need)
        return dfa::set_error(DFA_ERR_WORKSPACE, "dfa_ring_fwd: workspace must be 256-byte "
                              "aligned and hold %zu bytes", need);
    for (int p = 0; p < P; ++p)
        if (!workers[p].q || !workers[p].k || !workers[p].v || !workers[p].kv_slots ||
            !workers[p].o || !workers[p].lse)
            return dfa::set_error(DFA_ERR_INVALID_ARG, "dfa_ring_fwd: worker %d has a NULL "
                                  "buffer", p);
    float* o_part = reinterpret_cast<float*>((char*)ws + 256);
    float* lse_part = reinterpret_cast<float*>((char*)ws + 256 + align256(rows * desc->d * 4));
    cudaStream_t cs = (cudaStream_t)compute_stream;
    cudaStream_t xs = (overlap && copy_stream) ? (cudaStream_t)copy_stream : cs;
    const bool two = xs != cs;
    EventPair ev;
    if (two) {
        cudaError_t e = cudaEventCreateWithFlags(&ev.comp, cudaEventDisableTiming);
        if (e == cudaSuccess)
            e = cudaEventCreateWithFlags(&ev.copy, cudaEventDisableTiming);
        // the first copies overwrite slots that earlier work on the compute
        // stream may still read: order them after it
        if (e == cudaSuccess)
            e = cudaEventRecord(ev.comp, cs);
        if (e == cudaSuccess)
            e = cudaStreamWaitEvent(xs, ev.comp, 0);
        if (e != cudaSuccess)
            return cuda_err(e, "event creation");
    }
    auto slot = [&](int p, int i, int kv) -> void* {
        return (char*)workers[p].kv_slots + ((size_t)(2 * i + kv)) * kv_bytes;
    };
    const void* cur_k[64];
    const void* cur_v[64];
    for (int p = 0; p < P; ++p) {
        cur_k[p] = workers[p].k;
        cur_v[p] = workers[p].v;
    }
    for (int s = 0; s < P; ++s) {
        // "send": worker p receives its predecessor's current K/V for step s+1
        if (s + 1 < P) {
            if (two && s > 0) {
                cudaError_t e = cudaStreamWaitEvent(xs, ev.comp, 0);  // slot last read at s-1
                if (e != cudaSuccess)
                    return cuda_err(e, "stream wait");
            }
            for (int p = 0; p < P; ++p) {
                const int from = (p - 1 + P) % P;
                cudaError_t e = cudaMemcpyAsync(slot(p, s % 2, 0), cur_k[from], kv_bytes,
                                                cudaMemcpyDeviceToDevice, xs);
                if (e == cudaSuccess)
                    e = cudaMemcpyAsync(slot(p, s % 2, 1), cur_v[from], kv_bytes,
                                        cudaMemcpyDeviceToDevice, xs);
                if (e != cudaSuccess)
                    return cuda_err(e, "K/V copy");
            }
            if (two) {
                cudaError_t e = cudaEventRecord(ev.copy, xs);
                if (e != cudaSuccess)
                    return cuda_err(e, "event record");
            }
        }
        // compute: worker p against the keys of worker (p - s) mod P
        for (int p = 0; p < P; ++p) {
            const dfa_chunk_pair pair = {maps[p], maps[(p - s + P) % P]};
            const dfa_ring_worker& w = workers[p];
            dfa_status st;
            if (s == 0) {
                st = dfa_chunk_fwd(desc, &pair, n, n, w.q, cur_k[p], cur_v[p], w.o, w.lse, ws, 256,
                                   cs);
            } else {
                st = dfa_chunk_fwd(desc, &pair, n, n, w.q, cur_k[p], cur_v[p], o_part, lse_part,
                                   ws, 256, cs);
                if (st == DFA_OK)
                    st = dfa_lse_merge((int64_t)rows, desc->d, 1, o_part, lse_part, w.o, w.lse, 1,
                                       1, cs);
            }
            if (st != DFA_OK)
                return st;
        }
        if (s + 1 < P) {
            if (two) {
                cudaError_t e = cudaEventRecord(ev.comp, cs);
                if (e == cudaSuccess)
                    e = cudaStreamWaitEvent(cs, ev.copy, 0);  // next K/V has landed
                if (e != cudaSuccess)
                    return cuda_err(e, "event");
            }
            for (int p = 0; p < P; ++p) {
                cur_k[p] = slot(p, s % 2, 0);
                cur_v[p] = slot(p, s % 2, 1);
            }
        }
    }
    return DFA_OK;
}
