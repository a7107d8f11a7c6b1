/*
 * dfa.h -- C ABI of libdfa: exact causal blockwise attention (forward and
 * recomputation backward), chunk-pair partials, log-sum-exp merge, sequence
 * permutes and ring schedules, for NVIDIA GB300 (sm_103a).
 *
 * Conventions shared by every call
 * --------------------------------
 * - Tensors are row-major [B, H, L, d] (batch, head, token, feature),
 *   contiguous, on the device, 16-byte aligned.  Q, K, V, O, dO, dQ, dK, dV
 *   are bf16 unless a call says fp32.  LSE and D are fp32 [B, H, L].
 * - d (head dimension) is 64 or 128.  Hq % Hkv == 0; query head h reads
 *   key/value head h / (Hq / Hkv) (grouped-query attention).
 * - LSE is the natural-log log-sum-exp of the scaled, masked scores of a row:
 *   LSE_i = ln sum_j exp(scale * q_i . k_j).  A row that sees no key has
 *   LSE = -inf and O = 0.
 * - Causal masking is by global token position: key j is visible to query i
 *   iff pos(j) <= pos(i) (the diagonal is visible).
 * - Every call is asynchronous on the caller's CUDA stream (passed as void*,
 *   a cudaStream_t; NULL = legacy default stream).  No call allocates device
 *   memory or synchronises the device, except dfa_stream_status, which
 *   synchronises the given stream.  The caller owns every buffer; the library
 *   keeps no pointer after a call returns.
 * - Errors: argument errors are reported synchronously through the return
 *   value (no work is launched); launch failures return DFA_ERR_CUDA; a
 *   device-side wait that exceeds its time limit sets a status word in the
 *   workspace, read back by dfa_stream_status (DFA_ERR_TIMEOUT).  The text
 *   of the last error of the calling thread is in dfa_last_error().
 * - Workspace: calls that take (ws, ws_bytes) need at least
 *   dfa_workspace_size(desc, op) bytes, 256-byte aligned, whose first 256
 *   bytes (the status word) the caller zeroes once when allocating it.
 *   Workspace contents other than the status word are scratch.
 *
 * Sources of the method (web pages):
 * - "Striped Attention Guide: Faster Causal Ring Attention": "The Fatal Flaw:
 *   Causal Workload Imbalance" (causal score matrix), "Incremental Online
 *   Softmax Rescaling" (running max, sum, rescale of partial states),
 *   "Intra-Block vs. Inter-Block Masking Logic" (full / diagonal / skipped
 *   tiles), "Mathematical Formulation of Token Striping" and "Workload
 *   Balance Theorem" (striped partition, ring steps).
 * - "DistFlashAttn Guide: Distributed Attention for Long LLMs": "The Folded
 *   Chunk Assignment" (load-balanced partition), "The Causal Imbalance
 *   Crisis" (contiguous ring bubble and eta_util).
 * - "FlashAttention" glossary entry: tiled exact attention, O(N) memory, the
 *   backward pass recomputed from per-row softmax statistics.
 */
#ifndef DFA_H
#define DFA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum dfa_status {
    DFA_OK = 0,
    DFA_ERR_INVALID_ARG = 1, /* null pointer, bad size, inconsistent shape   */
    DFA_ERR_UNSUPPORTED = 2, /* valid but not implemented (d, alignment, map) */
    DFA_ERR_WORKSPACE = 3,   /* workspace missing or smaller than required    */
    DFA_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed             */
    DFA_ERR_TIMEOUT = 5,     /* a device-side wait gave up (async, see above) */
    DFA_ERR_BOUNDS = 6       /* a device-side index outside its tensor: only a
                                library built with DFA_DEBUG_BOUNDS checks and
                                reports this (async, like DFA_ERR_TIMEOUT)    */
} dfa_status;

/* Sequence partitions over P logical workers (chunks). */
enum {
    DFA_PART_CONTIGUOUS = 0, /* worker p: tokens [p n, (p+1) n), n = N / P   */
    DFA_PART_BALANCED = 1,   /* 2P chunks of N/(2P); worker p: chunk p then
                                chunk 2P-1-p (DistFlashAttn folded)          */
    DFA_PART_STRIPED = 2     /* blocks of `stripe` tokens dealt round-robin:
                                worker p owns blocks b with b mod P == p      */
};

/* Problem descriptor (plain data, caller-owned). */
typedef struct dfa_attn_desc {
    int32_t B;         /* batch                                            */
    int32_t Hq;        /* query heads                                      */
    int32_t Hkv;       /* key/value heads, Hq % Hkv == 0                   */
    int64_t N;         /* tokens per sequence                              */
    int32_t d;         /* head dimension, 64 or 128                        */
    int32_t causal;    /* 1 causal, 0 full attention                       */
    float scale;       /* softmax scale, usually 1/sqrt(d)                 */
    int32_t P;         /* logical workers (chunks), >= 1, N % P == 0        */
    int32_t partition; /* DFA_PART_*                                       */
    int32_t stripe;    /* striped block size in tokens (1 = token stripes) */
    int32_t o_fp32;    /* dfa_attn_fwd output O: 0 bf16, 1 fp32            */
    int32_t ndocs;     /* documents packed in the sequence (0: none)       */
    const int64_t* doc_bounds; /* device, ndocs + 1 increasing positions:
                                  document t is [doc_bounds[t],
                                  doc_bounds[t+1]), doc_bounds[0] = 0,
                                  doc_bounds[ndocs] = N.  A key is visible
                                  only to queries of its own document
                                  (Striped Attention Guide, "Document Packing
                                  and Boundary Alignment"); causal masking
                                  applies on top.  Not read by dfa_decode,
                                  which rejects ndocs != 0.               */
} dfa_attn_desc;

/*
 * Global positions of the rows of a chunk.  The chunk's rows form nseg (1 or
 * 2) segments; local row m' of segment t (m' counted from the segment start)
 * has position  base[t] + (m' / blk) * blk_stride + (m' % blk).
 * Positions must increase strictly along the chunk (blk_stride >= blk, and
 * base[1] above the last position of segment 0).
 *   contiguous worker p:  nseg 1, base p n, blk 1, blk_stride 1
 *   folded worker p:      nseg 2, len n/2 each, bases p n/2 and (2P-1-p) n/2
 *   striped worker p:     nseg 1, base p s, blk s, blk_stride P s
 */
typedef struct dfa_pos_map {
    int32_t nseg;
    int32_t reserved;
    int64_t len[2];
    int64_t base[2];
    int64_t blk;
    int64_t blk_stride;
} dfa_pos_map;

typedef struct dfa_chunk_pair {
    dfa_pos_map q;  /* positions of the query chunk's rows     */
    dfa_pos_map kv; /* positions of the key/value chunk's rows */
} dfa_chunk_pair;

/* Operations for dfa_workspace_size. */
enum { DFA_OP_FWD = 0, DFA_OP_BWD = 1, DFA_OP_CHUNK_FWD = 2, DFA_OP_CHUNK_BWD = 3,
       DFA_OP_RING_FWD = 4 };

/*
 * dfa_attn_fwd -- attention forward over a whole sequence (FlashAttention
 * glossary entry; Striped Attention Guide, "Incremental Online Softmax
 * Rescaling" and "Intra-Block vs. Inter-Block Masking Logic").
 *
 * Storage order: q/k/v/o/lse rows are in worker-major order of desc's
 * partition -- row r = p*n + m holds the token at global position
 * pos_p(m) (n = N/P).  With P == 1 or DFA_PART_CONTIGUOUS this is natural
 * order.  dfa_permute converts between natural and worker-major order.
 * One launch runs every ring step of every worker: worker p's queries meet
 * the keys of worker (p - s) mod P for s = 0..P-1, fully masked tiles are
 * skipped, and the per-step partial states are merged on chip by the same
 * log-sum-exp rescaling that dfa_lse_merge applies in memory.
 *   q [B,Hq,N,d] bf16, k/v [B,Hkv,N,d] bf16  (inputs)
 *   o [B,Hq,N,d] bf16 (desc->o_fp32 == 0) or fp32 (== 1), lse [B,Hq,N] fp32
 *   ws: dfa_workspace_size(desc, DFA_OP_FWD) bytes.
 */
dfa_status dfa_attn_fwd(const dfa_attn_desc* desc, const void* q, const void* k,
                        const void* v, void* o, float* lse, void* ws, size_t ws_bytes,
                        void* stream);

/*
 * dfa_attn_bwd -- recomputation backward of dfa_attn_fwd (FlashAttention
 * glossary entry: scores are recomputed from Q, K and the per-row LSE instead
 * of stored).  Same storage order as dfa_attn_fwd.  With D_i = dO_i . O_i,
 * P = exp(scale Q K^T - LSE):  dV = P^T dO,  dS = P o (dO V^T - D),
 * dQ = scale dS K,  dK = scale dS^T Q  (dK, dV summed over the Hq/Hkv query
 * heads of a key/value head).
 *   o [B,Hq,N,d] bf16 (the forward output), dout [B,Hq,N,d] bf16,
 *   lse [B,Hq,N] fp32 (the forward's);  dq [B,Hq,N,d], dk/dv [B,Hkv,N,d] bf16.
 *   ws: dfa_workspace_size(desc, DFA_OP_BWD) bytes: the fp32 dQ accumulator
 *   and, per query row, 32-byte records of -LSE/scale and -D that the
 *   kernel adds to S and dP on the tensor core; when N * Hq/Hkv > 131072
 *   also fp32
 *   dK and dV, which the kernel sums over blocks of query rows before the
 *   bf16 conversion.
 */
dfa_status dfa_attn_bwd(const dfa_attn_desc* desc, const void* q, const void* k,
                        const void* v, const void* o, const void* dout, const float* lse,
                        void* dq, void* dk, void* dv, void* ws, size_t ws_bytes,
                        void* stream);

/*
 * dfa_chunk_fwd -- one chunk pair: a query chunk against a key/value chunk at
 * the global positions given by pair (Striped Attention Guide, "Incremental
 * Online Softmax Rescaling", steps 1-2: scores of the local queries against
 * the current key block, masked where GlobalPos(q) < GlobalPos(k)).
 * Produces the normalised partial of that pair: o_part = softmax over the
 * pair's visible keys times V, lse_part its log-sum-exp; rows that see no key
 * of the chunk get (0, -inf).  desc supplies B, Hq, Hkv, d, causal, scale.
 *   q [B,Hq,Lq,d] bf16, k/v [B,Hkv,Lk,d] bf16;
 *   o_part [B,Hq,Lq,d] fp32, lse_part [B,Hq,Lq] fp32.
 *   Lq, Lk must equal the total lengths of pair->q and pair->kv.
 */
dfa_status dfa_chunk_fwd(const dfa_attn_desc* desc, const dfa_chunk_pair* pair, int64_t Lq,
                         int64_t Lk, const void* q, const void* k, const void* v,
                         float* o_part, float* lse_part, void* ws, size_t ws_bytes,
                         void* stream);

/*
 * dfa_chunk_bwd -- gradient contribution of one chunk pair to the attention
 * over the whole sequence.  lse must be the MERGED (whole-sequence) LSE of the
 * query rows and delta their D_i = dO_i . O_i with the final O; when delta is
 * NULL it is computed here from o and dout (o bf16 [B,Hq,Lq,d]).
 * Accumulates (+=) into fp32 dq_acc [B,Hq,Lq,d], dk_acc / dv_acc
 * [B,Hkv,Lk,d]; the caller zeroes them before the first pair.  dq_acc and
 * dk_acc include the softmax scale.
 *   ws: dfa_workspace_size(desc, DFA_OP_CHUNK_BWD) bytes with desc->N = Lq
 *   (per query row the 32-byte -LSE/scale and -D records).
 */
dfa_status dfa_chunk_bwd(const dfa_attn_desc* desc, const dfa_chunk_pair* pair, int64_t Lq,
                         int64_t Lk, const void* q, const void* k, const void* v,
                         const void* o, const void* dout, const float* lse,
                         const float* delta, float* dq_acc, float* dk_acc, float* dv_acc,
                         void* ws, size_t ws_bytes, void* stream);

/*
 * dfa_lse_merge -- merge k partial results of the same rows by log-sum-exp
 * rescaling (Striped Attention Guide, "Incremental Online Softmax
 * Rescaling", the alpha/beta update written for normalised partials):
 *   LSE = ln sum_c exp(LSE_c),   O = sum_c exp(LSE_c - LSE) O_c.
 * A row whose partials are all -inf gives (0, -inf), never NaN.
 *   o_parts [k][rows][d] fp32, lse_parts [k][rows] fp32 (read only)
 *   o_out [rows][d] fp32 (out_fp32 = 1) or bf16 (0); lse_out [rows] fp32.
 *   accumulate = 1: (o_out, lse_out) is itself a partial and is merged in
 *   (in place; requires out_fp32 = 1).  k >= 1, or k = 0 with accumulate.
 */
dfa_status dfa_lse_merge(int64_t rows, int32_t d, int32_t k, const float* o_parts,
                         const float* lse_parts, void* o_out, float* lse_out,
                         int32_t out_fp32, int32_t accumulate, void* stream);

/*
 * dfa_ring_fwd -- the ring schedule of context-parallel attention on one GPU
 * (DistFlashAttn Guide, the ring over P workers; Striped Attention Guide,
 * "Workload Balance Theorem": at ring step s worker p holds the key/value
 * chunk of worker (p - s) mod P, and "Incremental Online Softmax Rescaling":
 * each step's partial is merged into the worker's running result).
 * Worker p holds chunk p of desc's partition (P workers, chunks of n = N/P
 * tokens, in worker-major order as dfa_permute produces them).  At each of
 * the P steps every worker runs dfa_chunk_fwd against the K/V chunk it
 * holds and merges the partial into its (o, lse) with dfa_lse_merge; the
 * hand-over of K/V to the next worker is a device-to-device copy into one of
 * the receiver's two slots, issued on copy_stream while the step computes
 * (overlap = 1), or on compute_stream before it (overlap = 0, for timing the
 * difference).  The result equals attention over the whole sequence.
 *   workers[p].q [B,Hq,n,d], .k/.v [B,Hkv,n,d] bf16 (read only);
 *   .kv_slots 4 * B*Hkv*n*d bf16 (the two receive slots, K then V each);
 *   .o [B,Hq,n,d] fp32 and .lse [B,Hq,n] fp32 (written).
 *   ws: dfa_workspace_size(desc, DFA_OP_RING_FWD) bytes (a partial's O, LSE).
 * Both streams are the caller's; when the call returns all work is ordered
 * before later work on compute_stream.
 */
typedef struct dfa_ring_worker {
    const void* q;
    const void* k;
    const void* v;
    void* kv_slots;
    float* o;
    float* lse;
} dfa_ring_worker;

dfa_status dfa_ring_fwd(const dfa_attn_desc* desc, const dfa_ring_worker* workers, void* ws,
                        size_t ws_bytes, int32_t overlap, void* compute_stream,
                        void* copy_stream);

/*
 * dfa_attn_step_host -- one training step of attention with its tensors in
 * HOST memory, in natural token order: the permute into desc's worker-major
 * order, dfa_attn_fwd, dfa_attn_bwd and the permutes back (the forward and
 * recomputation backward of the FlashAttention glossary entry over the
 * partition of desc), with the host-to-device and device-to-host copies
 * inside the call.  The pages describe no counterpart: this is the
 * library's host-streaming executor.
 *
 * The work is cut into groups of kv_heads_per_group key/value heads of one
 * batch item, each with its Hq/Hkv query heads (heads never interact, so a
 * group is a complete problem of B = 1).  Group g's upload (h2d_stream), its
 * compute (compute_stream) and its download (d2h_stream) are ordered by
 * events, so that group g+1 uploads and group g-1 downloads while group g
 * computes; device staging is double-buffered in ws.  When either copy
 * stream is given, odd groups compute on a stream the call creates (and
 * releases) and even groups on compute_stream, so that a group's forward
 * starts on the SMs the previous group's backward releases; the backwards
 * themselves run one after another.  With pinned host memory the copies
 * overlap the compute; pageable memory gives the same results with the
 * copies serialised by the driver.  h2d_stream or d2h_stream NULL: those
 * copies run on compute_stream, in order (and with both NULL, everything
 * runs on compute_stream).
 *   h_q, h_dout [B,Hq,N,d] bf16; h_k, h_v [B,Hkv,N,d] bf16 (read);
 *   h_o, h_dq [B,Hq,N,d] bf16, h_lse [B,Hq,N] fp32, h_dk, h_dv [B,Hkv,N,d]
 *   bf16 (written; O is the forward output, LSE its natural-log row
 *   log-sum-exp).  Host buffers must stay valid and untouched until
 *   compute_stream has passed the call's work.
 *   kv_heads_per_group: a divisor of Hkv, or 0 for the library's choice
 *   (the fewest heads per group that still give the group's backward at
 *   least 2432 key tiles of 128 rows, and at least two groups where B*Hkv
 *   allows).  With the library's choice, groups of 4 or more heads, the
 *   call's first and last groups are each cut into a quarter and three
 *   quarters (the quarter first at the start, last at the end): the first
 *   upload and the last download, which no compute overlaps, then move a
 *   quarter of a group.
 *   ws: dfa_attn_step_host_workspace_size(desc, kv_heads_per_group) bytes,
 *   status word first (dfa_stream_status reads the backward's timeouts).
 * desc->o_fp32 must be 0 (DFA_ERR_UNSUPPORTED otherwise).  When the call
 * returns, all of its work, on every stream, is ordered before later work
 * on compute_stream; an error returned after work was queued still orders
 * the queued work so.
 */
size_t dfa_attn_step_host_workspace_size(const dfa_attn_desc* desc,
                                         int32_t kv_heads_per_group);
dfa_status dfa_attn_step_host(const dfa_attn_desc* desc, const void* h_q, const void* h_k,
                              const void* h_v, const void* h_dout, void* h_o, float* h_lse,
                              void* h_dq, void* h_dk, void* h_dv, int32_t kv_heads_per_group,
                              void* ws, size_t ws_bytes, void* compute_stream,
                              void* h2d_stream, void* d2h_stream);

/*
 * dfa_attn_steps_host -- nsteps consecutive steps of dfa_attn_step_host in
 * one call (at most 64): the same work and results as nsteps calls, but the
 * (step, group) items form one stream, so the first groups of step t + 1
 * upload while the last groups of step t compute and download.  Only the
 * first upload and the last download of the whole call are left unhidden.
 * steps[t] holds step t's host tensors, with the layouts and rules of
 * dfa_attn_step_host (the same buffers may serve several steps when the
 * caller expects them to be overwritten in step order).  Same workspace as
 * dfa_attn_step_host.  The pages describe no counterpart: this is the
 * host-streaming executor's loop over training steps.
 */
typedef struct dfa_host_step {
    const void* q;
    const void* k;
    const void* v;
    const void* dout;
    void* o;
    float* lse;
    void* dq;
    void* dk;
    void* dv;
} dfa_host_step;

dfa_status dfa_attn_steps_host(const dfa_attn_desc* desc, int32_t nsteps,
                               const dfa_host_step* steps, int32_t kv_heads_per_group,
                               void* ws, size_t ws_bytes, void* compute_stream,
                               void* h2d_stream, void* d2h_stream);

/*
 * dfa_decode -- split-KV decoding: T query tokens per sequence against L
 * cached keys (FlashAttention glossary entry, the Flash-Decoding variant:
 * the keys are cut into splits of split_len, each split gives a normalised
 * partial (O, LSE) on its own CTAs, and the partials are merged by the LSE
 * rescaling of dfa_lse_merge).  Query token t sits at position q_pos0 + t,
 * cached key j at position j; with desc->causal, key j is visible to token t
 * iff j <= q_pos0 + t.  desc supplies B, Hq, Hkv, d, causal, scale, o_fp32.
 *   q [B,Hq,T,d] bf16; k, v [B,Hkv,L,d] bf16;
 *   o [B,Hq,T,d] bf16 (o_fp32 = 0) or fp32; lse [B,Hq,T] fp32.
 *   split_len: a positive multiple of 64; (Hq/Hkv) * T <= 16.
 *   ws: dfa_decode_workspace_size(desc, T, L, split_len) bytes (partials).
 * The split partials run on CUDA cores (every K/V row is read once and meets
 * a handful of query rows: memory-bound, not a tensor-core contraction).
 */
size_t dfa_decode_workspace_size(const dfa_attn_desc* desc, int32_t T, int64_t L,
                                 int32_t split_len);
dfa_status dfa_decode(const dfa_attn_desc* desc, int32_t T, int64_t L, int64_t q_pos0,
                      const void* q, const void* k, const void* v, void* o, float* lse,
                      int32_t split_len, void* ws, size_t ws_bytes, void* stream);

/*
 * dfa_permute -- gather rows between natural order and the worker-major order
 * of desc's partition (Striped Attention Guide, the partitioner's
 * stripe/unstripe; DistFlashAttn Guide, "The Folded Chunk Assignment").
 * in/out are [heads][N][row_elems] with elements of elem_bytes (2 or 4).
 * inverse = 0: out[h][p n + m] = in[h][pos_p(m)];  inverse = 1: the reverse.
 * in and out must not overlap.  row_elems * elem_bytes must be a multiple of 4.
 */
dfa_status dfa_permute(const dfa_attn_desc* desc, int32_t inverse, const void* in, void* out,
                       int32_t elem_bytes, int64_t row_elems, int64_t heads, void* stream);

/*
 * dfa_permute_rope -- dfa_permute of bf16 query or key rows fused with the
 * rotary position embedding at each token's global position (Striped
 * Attention Guide, "Preserving Rotary Position Embeddings": token i is
 * rotated by R(Theta, i) using its absolute index, i = m P + p for a
 * token-striped worker p, before the ring, so that rotated inner products
 * depend only on i - j whatever the storage order).
 * Rotation: feature pairs (2t, 2t+1), t < d/2, turned by the angle
 * i * theta_base^(-2t/d) (x' = x cos - y sin, y' = x sin + y cos), computed
 * in fp32 after an fp64 reduction of the angle, rounded to bf16.
 *   in, out: [heads, N, d] bf16 (d = desc->d), 16-byte aligned, not
 *   overlapping; heads = B * H.  inverse = 0: natural order in, worker-major
 *   order out, rotation by +angle; inverse = 1: worker-major in, natural out,
 *   rotation by -angle (the transpose, for gradients dQ and dK).
 *   theta_base: > 1 (10000 for Llama-7B).
 * Returns DFA_ERR_INVALID_ARG on a bad descriptor, NULL or overlapping
 * buffers or a bad base, DFA_ERR_UNSUPPORTED on misaligned pointers.
 */
dfa_status dfa_permute_rope(const dfa_attn_desc* desc, int32_t inverse, const void* in,
                            void* out, int64_t heads, float theta_base, void* stream);

/*
 * Ring schedule (host only, no device work) for the P workers of desc's
 * partition (Striped Attention Guide, "Workload Balance Theorem": at ring
 * step s worker p holds the keys of worker (p - s) mod P; "Intra-Block vs.
 * Inter-Block Masking Logic": a tile pair is skipped, computed without a mask
 * or computed with an element mask; DistFlashAttn Guide, "The Causal
 * Imbalance Crisis" and "The Folded Chunk Assignment").  Causal masking by
 * global position only: desc's documents are not taken into account.
 *
 * The query rows of a worker's chunk are cut into tiles of tile_m rows, the
 * key rows into tiles of tile_n rows (the last tile of each may be short).
 * Because positions increase along every chunk, the key tiles that a query
 * tile sees form a prefix of the key chunk, and the ones it sees without a
 * mask a shorter prefix; so the tile pairs of a query tile are at most three
 * work items, each a range of key tiles of one class:
 *   DFA_TILE_FULL     [0, full)      every (query, key) pair visible
 *   DFA_TILE_PARTIAL  [full, vis)    an element mask is needed
 *   DFA_TILE_SKIP     [vis, nkt)     no pair visible (never computed)
 * (non-causal: one FULL item [0, nkt)).  Empty ranges give no item.
 *
 * Outputs (all caller-owned host memory; any array pointer may be NULL to
 * skip that output):
 *   pair_tokens[p*P + s]     visible (query, key) token pairs of worker p at
 *                            step s;
 *   tile_counts[(p*P + s)*3 + c]  tiles of class c (0 skip, 1 full,
 *                            2 partial) of that pair;
 *   pairs[p*P + s]           the pair list: worker, step, the key/value
 *                            worker it holds, its tokens and the range of
 *                            its work items in items[];
 *   items[0 .. n_items)      the tile work items, pair by pair (p major,
 *                            then s), query tile by query tile, in class
 *                            order FULL, PARTIAL, SKIP;
 *   total_pairs, eta_slots = non-empty (p, s) slots / P^2 (the pages'
 *   eta_util), eta_flops = total pairs / (P * sum_s max_p pair_tokens)
 *   (lockstep utilisation).
 * Item buffer protocol: n_items is always set to the number of items the
 * schedule has.  capacity = 0 (or items = NULL) is a size query: nothing is
 * written to items.  0 < capacity < n_items returns DFA_ERR_INVALID_ARG.
 */
enum { DFA_TILE_SKIP = 0, DFA_TILE_FULL = 1, DFA_TILE_PARTIAL = 2 };

typedef struct dfa_sched_pair {
    int32_t worker;     /* p: holds the query chunk of worker p            */
    int32_t step;       /* s: ring step                                    */
    int32_t kv_worker;  /* (p - s) mod P: whose keys/values it holds        */
    int32_t reserved;
    int64_t tokens;     /* visible (query, key) token pairs                */
    int64_t first_item; /* index of the pair's first item in items[]       */
    int64_t n_items;    /* number of items of the pair                     */
} dfa_sched_pair;

typedef struct dfa_sched_item {
    int32_t worker, step; /* the pair                                      */
    int32_t q_tile;       /* query tile index inside the worker's chunk    */
    int32_t kv_begin;     /* key tile range [kv_begin, kv_end) inside the  */
    int32_t kv_end;       /*   key/value chunk                             */
    int32_t mask_class;   /* DFA_TILE_FULL / DFA_TILE_PARTIAL / DFA_TILE_SKIP */
} dfa_sched_item;

typedef struct dfa_schedule {
    int64_t* pair_tokens;   /* [P*P] or NULL                               */
    int64_t* tile_counts;   /* [P*P*3] or NULL                             */
    int64_t total_pairs;
    double eta_slots;
    double eta_flops;
    dfa_sched_pair* pairs;  /* [P*P] or NULL                               */
    dfa_sched_item* items;  /* [capacity] or NULL                          */
    int64_t capacity;       /* in: items[] capacity (0: size query)        */
    int64_t n_items;        /* out: items of the schedule                  */
} dfa_schedule;

dfa_status dfa_make_schedule(const dfa_attn_desc* desc, int32_t tile_m, int32_t tile_n,
                             dfa_schedule* out);

/* The position map of worker p under desc's partition (host only). */
dfa_status dfa_partition_map(const dfa_attn_desc* desc, int32_t p, dfa_pos_map* out);

/*
 * dfa_attn_bwd_noalloc -- dfa_attn_bwd for callers that cannot allocate device
 * memory.  The pages describe no counterpart: this is a library convenience.
 *
 * Who needs it: code that has tensor pointers but no allocator it may use --
 * a plugin handed buffers by a host framework, a host callback, a loop that
 * forbids cudaMalloc after start-up.  dfa_attn_bwd needs a workspace of
 * dfa_workspace_size(desc, DFA_OP_BWD) bytes (256 + B*Hq*N*(4d + 64),
 * rounded, plus 8*B*Hkv*N*d when N * Hq/Hkv > 131072); here that scratch is
 * a fixed 64 MiB array in device memory owned by the library, held
 * by every GPU that loads the library until the process exits.  Problems
 * whose scratch would exceed 64 MiB are rejected with DFA_ERR_WORKSPACE.
 *
 * Same arguments, layouts and results as dfa_attn_bwd, minus the workspace.
 * This call allocates nothing.  Its first call on a device looks up the
 * array's device address (with that device current), so make that first call
 * before any stream capture.  All calls on a device share the array and it
 * keeps the last call's contents: calls that overlap on the GPU (unordered
 * streams) race.  A device-side wait timeout of this call is recorded in the
 * shared array, not in a caller workspace, so dfa_stream_status cannot report
 * it; the call's outputs are then invalid.
 */
dfa_status dfa_attn_bwd_noalloc(const dfa_attn_desc* desc, const void* q, const void* k,
                                const void* v, const void* o, const void* dout,
                                const float* lse, void* dq, void* dk, void* dv, void* stream);

/* Bytes of workspace that op needs for desc (0 on invalid arguments). */
size_t dfa_workspace_size(const dfa_attn_desc* desc, int32_t op);

/*
 * Synchronise stream, then read and clear the device status word in ws.
 * Returns DFA_OK, DFA_ERR_TIMEOUT (a kernel gave up waiting; its outputs are
 * invalid), DFA_ERR_BOUNDS (bounds-checking build only: a kernel computed an
 * index outside a tensor and skipped that access) or DFA_ERR_CUDA (the
 * stream reported an error).
 */
dfa_status dfa_stream_status(void* ws, void* stream);

/*
 * Self-test of the bounded-wait path: launches one block that waits on a
 * barrier nothing will complete, with a limit of timeout_us microseconds;
 * the wait gives up, records DFA_ERR_TIMEOUT in ws and the kernel returns.
 */
dfa_status dfa_selftest_timeout(void* ws, int64_t timeout_us, void* stream);

const char* dfa_status_string(dfa_status s);
const char* dfa_last_error(void);
int32_t dfa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DFA_H */
