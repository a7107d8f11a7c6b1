// dfa_mem.cu -- the bandwidth-bound kernels: log-sum-exp merge of partial
// results, sequence permutes between natural and worker-major order (plain, or
// with the rotary embedding at global positions), the backward preprocess
// (D = rowsum(dO * O), the row-constant records, zeroing the dQ accumulator), the
// dQ fp32 -> bf16 conversion, and the bounded-wait self-test.
//
// All are grid-stride loops over 16-byte vectors with several independent
// loads in flight per thread; grids are a multiple of the SM count.
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "dfa_params.h"
#include "dfa_ptx.cuh"

namespace dfa {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;

// ---------------------------------------------------------------------------
// LSE merge (Striped Attention Guide, "Incremental Online Softmax Rescaling":
// the alpha/beta rescale of partial states, for normalised partials):
//   LSE = m + ln sum_c exp(LSE_c - m),  O = sum_c exp(LSE_c - LSE) O_c.
// TPR = d/4 threads per row, one float4 of each partial per thread.
// ---------------------------------------------------------------------------
template <int D, bool OUT_F32, bool ACC>
__global__ void __launch_bounds__(256, 4) lse_merge_kernel(int64_t rows, int k,
                                                        const float* __restrict__ o_parts,
                                                        const float* __restrict__ lse_parts,
                                                        void* __restrict__ o_out,
                                                        float* __restrict__ lse_out)
{
    constexpr int TPR = D / 4;
    constexpr int RPB = 256 / TPR;  // rows per block iteration
    const int sub = threadIdx.x % TPR;
    const int64_t row_base = (int64_t)blockIdx.x * RPB + threadIdx.x / TPR;
    const int64_t row_step = (int64_t)gridDim.x * RPB;
    for (int64_t r = row_base; r < rows; r += row_step) {
        float m = -INFINITY;
        float lacc = -INFINITY;
        if (ACC) {
            lacc = lse_out[r];
            m = lacc;
        }
        for (int c = 0; c < k; ++c)
            m = fmaxf(m, __ldg(lse_parts + (int64_t)c * rows + r));
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        float lse = -INFINITY;
        if (m != -INFINITY) {
            const float mb = m * kLog2e;
            float sum = 0.f;
            if (ACC) {
                const float w = ex2(fmaf(lacc, kLog2e, -mb));
                const float4 v = reinterpret_cast<const float4*>(
                    reinterpret_cast<float*>(o_out) + r * D)[sub];
                sum += w;
                acc.x = w * v.x;
                acc.y = w * v.y;
                acc.z = w * v.z;
                acc.w = w * v.w;
            }
            int c = 0;
            for (; c + 4 <= k; c += 4) {
                float w[4];
                float4 v[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    w[i] = __ldg(lse_parts + (int64_t)(c + i) * rows + r);
                    v[i] = __ldg(reinterpret_cast<const float4*>(
                                     o_parts + ((int64_t)(c + i) * rows + r) * D) +
                                 sub);
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float e = ex2(fmaf(w[i], kLog2e, -mb));
                    sum += e;
                    acc.x = fmaf(e, v[i].x, acc.x);
                    acc.y = fmaf(e, v[i].y, acc.y);
                    acc.z = fmaf(e, v[i].z, acc.z);
                    acc.w = fmaf(e, v[i].w, acc.w);
                }
            }
            for (; c < k; ++c) {
                const float e = ex2(fmaf(__ldg(lse_parts + (int64_t)c * rows + r), kLog2e, -mb));
                const float4 v = __ldg(
                    reinterpret_cast<const float4*>(o_parts + ((int64_t)c * rows + r) * D) + sub);
                sum += e;
                acc.x = fmaf(e, v.x, acc.x);
                acc.y = fmaf(e, v.y, acc.y);
                acc.z = fmaf(e, v.z, acc.z);
                acc.w = fmaf(e, v.w, acc.w);
            }
            const float inv = 1.f / sum;
            acc.x *= inv;
            acc.y *= inv;
            acc.z *= inv;
            acc.w *= inv;
            lse = m + lg2(sum) * kLn2;
        }
        if (OUT_F32) {
            reinterpret_cast<float4*>(reinterpret_cast<float*>(o_out) + r * D)[sub] = acc;
        } else {
            uint2 pk = make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
            reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(o_out) + r * D)[sub] = pk;
        }
        if (sub == 0)
            lse_out[r] = lse;
    }
}

cudaError_t launch_lse_merge(int64_t rows, int d, int k, const float* o_parts,
                             const float* lse_parts, void* o_out, float* lse_out, int out_fp32,
                             int accumulate, int num_sms, cudaStream_t stream)
{
    const int rpb = 256 / (d / 4);
    int64_t blocks = (rows + rpb - 1) / rpb;
    const int64_t cap = (int64_t)num_sms * 8;
    if (blocks > cap)
        blocks = cap;
    if (blocks < 1)
        blocks = 1;
#define DFA_MERGE(DD, F32, ACC)                                                              \
    lse_merge_kernel<DD, F32, ACC><<<(int)blocks, 256, 0, stream>>>(rows, k, o_parts, lse_parts, \
                                                                     o_out, lse_out)
    if (d == 128) {
        if (accumulate)
            DFA_MERGE(128, true, true);
        else if (out_fp32)
            DFA_MERGE(128, true, false);
        else
            DFA_MERGE(128, false, false);
    } else {
        if (accumulate)
            DFA_MERGE(64, true, true);
        else if (out_fp32)
            DFA_MERGE(64, true, false);
        else
            DFA_MERGE(64, false, false);
    }
#undef DFA_MERGE
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Permute: out[h][p n + m] = in[h][pos_p(m)] (inverse swaps the roles).
// VEC bytes per thread step (16 or 4); row_vecs vectors per row.
// ---------------------------------------------------------------------------
template <typename V>
__global__ void __launch_bounds__(256) permute_kernel(const __grid_constant__ PermuteParams p,
                                                      const V* __restrict__ in,
                                                      V* __restrict__ out)
{
    const int64_t per_head = (int64_t)p.N * p.row_vecs;
    const int64_t total = p.heads * per_head;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t h = i / per_head;
        const int64_t rem = i - h * per_head;
        const int32_t r = (int32_t)(rem / p.row_vecs);  // worker-major row
        const int32_t v = (int32_t)(rem - (int64_t)r * p.row_vecs);
        const int32_t w = r / p.n, m = r - w * p.n;
        const int32_t g = map_pos(p.map[w], m);         // natural row
        const int64_t wm = (h * p.N + r) * p.row_vecs + v;
        const int64_t nat = (h * p.N + g) * p.row_vecs + v;
        if (p.inverse)
            out[nat] = __ldg(in + wm);
        else
            out[wm] = __ldg(in + nat);
    }
}

cudaError_t launch_permute(const PermuteParams& pp, const void* in, void* out, int vec_bytes,
                           int num_sms, cudaStream_t stream)
{
    const int64_t total = pp.heads * (int64_t)pp.N * pp.row_vecs;
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = (int64_t)num_sms * 16;
    if (blocks > cap)
        blocks = cap;
    if (blocks < 1)
        blocks = 1;
    if (vec_bytes == 16)
        permute_kernel<uint4><<<(int)blocks, 256, 0, stream>>>(pp, (const uint4*)in, (uint4*)out);
    else
        permute_kernel<uint32_t>
            <<<(int)blocks, 256, 0, stream>>>(pp, (const uint32_t*)in, (uint32_t*)out);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Permute with rotary position embedding at the tokens' global positions
// (Striped Attention Guide, "Preserving Rotary Position Embeddings": the
// rotation R(Theta, i) of token i is applied with its absolute position i,
// i = m P + p for token-striped storage, before the ring).  Feature pairs
// (2t, 2t+1) are rotated by the angle i * theta_t; `inverse` applies the
// transposed rotation and the inverse permutation (the gradient path).
// ---------------------------------------------------------------------------
// One warp per token row at a time: lane l owns 16-byte vector v = l mod V
// (V = d/8 vectors per head row, 4 feature pairs each) of heads l div V,
// l div V + 32/V, ...; it reduces its own 4 angles (in fp64: i * theta_t
// reaches 5e5 radians at N = 512K, where an fp32 product would be off by up
// to 0.03), so no shared memory or block barrier is needed.
__global__ void __launch_bounds__(256) permute_rope_kernel(const __grid_constant__ RopeParams rp,
                                                           const uint4* __restrict__ in,
                                                           uint4* __restrict__ out)
{
    const PermuteParams& p = rp.perm;
    const int vecs = rp.d / 8;             // 8 or 16
    const int lane = threadIdx.x & 31;
    const int v = lane & (vecs - 1);
    const int h0 = lane / vecs, hstep = 32 / vecs;
    const int warps = gridDim.x * (blockDim.x >> 5);
    constexpr double kTwoPi = 6.283185307179586;
    for (int32_t r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < p.N; r += warps) {
        const int32_t w = r / p.n, m = r - w * p.n;
        const int32_t g = map_pos(p.map[w], m);  // natural row = global position
        float2 cs[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            // Cody-Waite style reduction of the angle into [-pi, pi] in fp64
            const double a = (double)g * rp.theta[4 * v + e];
            const double k = rint(a * (1.0 / kTwoPi));
            const float red = (float)fma(-k, kTwoPi, a);
            float sn, c;
            sincosf(red, &sn, &c);
            cs[e] = make_float2(c, p.inverse ? -sn : sn);
        }
#pragma unroll 4
        for (int64_t h = h0; h < p.heads; h += hstep) {
            const int64_t wm = (h * p.N + r) * vecs + v;
            const int64_t nat = (h * p.N + g) * vecs + v;
            const uint4 x = __ldg(in + (p.inverse ? wm : nat));
            uint32_t xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float a = bf16lo(xs[e]), b = bf16hi(xs[e]);
                xs[e] = pack_bf16x2(a * cs[e].x - b * cs[e].y, a * cs[e].y + b * cs[e].x);
            }
            out[p.inverse ? nat : wm] = make_uint4(xs[0], xs[1], xs[2], xs[3]);
        }
    }
}

cudaError_t launch_permute_rope(const RopeParams& rp, const void* in, void* out, int num_sms,
                                cudaStream_t stream)
{
    int64_t blocks = (rp.perm.N + 7) / 8;  // 8 warps per block, a row each
    const int64_t cap = (int64_t)num_sms * 8;
    if (blocks > cap)
        blocks = cap;
    if (blocks < 1)
        blocks = 1;
    permute_rope_kernel<<<(int)blocks, 256, 0, stream>>>(rp, (const uint4*)in, (uint4*)out);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Backward preprocess: D[r] = sum_c dO[r][c] * O[r][c] (fp32 accumulate) or
// the caller's D, the per-row records of -LSE/scale and -D for the tensor
// core, and dq_acc[r][:] = 0 when dq_acc is non-null.  D/8 threads per row,
// 16 bytes of each bf16 tensor per thread.
// ---------------------------------------------------------------------------
// One K = 16 slice record that adds x to a product through the tensor core:
// x split into three bf16 values hi + mid + lo (|x - hi - mid - lo| <= 2^-24
// |x|, the precision of fp32) at K positions 0, 1 and 8, zeros elsewhere;
// the matching operand row holds ones at K positions 0, 1, 8 and 9.
__device__ __forceinline__ void aug_record(float x, uint4* dst)
{
    const __nv_bfloat16 hi = __float2bfloat16_rn(x);
    const float r1 = x - __bfloat162float(hi);
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const __nv_bfloat16 lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
    dst[0] = make_uint4((uint32_t)__bfloat16_as_ushort(hi) |
                            ((uint32_t)__bfloat16_as_ushort(mid) << 16),
                        0u, 0u, 0u);
    dst[1] = make_uint4((uint32_t)__bfloat16_as_ushort(lo), 0u, 0u, 0u);
}

// Per row: D = dO . O (or the caller's delta), the records of -LSE/scale
// (0 for a row without keys, whose P is masked anyway) and -D, and zeroing
// of the fp32 dQ accumulator row.
template <int D>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(
    int64_t rows, const uint4* __restrict__ o, const uint4* __restrict__ dout,
    const float* __restrict__ delta, const float* __restrict__ lse, float inv_scale,
    uint4* __restrict__ aug_lse, uint4* __restrict__ aug_delta, float4* __restrict__ dq_acc)
{
    constexpr int TPR = D / 8;
    constexpr int RPB = 256 / TPR;
    const int sub = threadIdx.x % TPR;
    // the loop bound is block-uniform so that every lane reaches the shuffles
    for (int64_t rb = (int64_t)blockIdx.x * RPB; rb < rows; rb += (int64_t)gridDim.x * RPB) {
        const int64_t r = rb + threadIdx.x / TPR;
        const bool ok = r < rows;
        float s = 0.f;
        if (o) {
            const uint4 a = ok ? __ldg(o + r * TPR + sub) : make_uint4(0u, 0u, 0u, 0u);
            const uint4 b = ok ? __ldg(dout + r * TPR + sub) : make_uint4(0u, 0u, 0u, 0u);
            s = bf16lo(a.x) * bf16lo(b.x) + bf16hi(a.x) * bf16hi(b.x);
            s = fmaf(bf16lo(a.y), bf16lo(b.y), s);
            s = fmaf(bf16hi(a.y), bf16hi(b.y), s);
            s = fmaf(bf16lo(a.z), bf16lo(b.z), s);
            s = fmaf(bf16hi(a.z), bf16hi(b.z), s);
            s = fmaf(bf16lo(a.w), bf16lo(b.w), s);
            s = fmaf(bf16hi(a.w), bf16hi(b.w), s);
#pragma unroll
            for (int off = TPR / 2; off > 0; off >>= 1)
                s += __shfl_xor_sync(0xffffffffu, s, off);
        } else if (ok && sub == 0) {
            s = delta[r];
        }
        if (ok && sub == 0) {
            const float l = lse[r];
            aug_record(l == -INFINITY ? 0.f : -l * inv_scale, aug_lse + 2 * r);
            aug_record(-s, aug_delta + 2 * r);
        }
        if (ok && dq_acc) {
            const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
            dq_acc[r * (D / 4) + 2 * sub] = z;
            dq_acc[r * (D / 4) + 2 * sub + 1] = z;
        }
    }
}

cudaError_t launch_bwd_preprocess(int64_t rows, int d, const void* o, const void* dout,
                                  const float* delta, const float* lse, float scale,
                                  void* aug_lse, void* aug_delta, float* dq_acc, int num_sms,
                                  cudaStream_t stream)
{
    const int rpb = 256 / (d / 8);
    int64_t blocks = (rows + rpb - 1) / rpb;
    const int64_t cap = (int64_t)num_sms * 8;
    if (blocks > cap)
        blocks = cap;
    if (blocks < 1)
        blocks = 1;
    const float inv = 1.f / scale;
    if (d == 128)
        bwd_preprocess_kernel<128><<<(int)blocks, 256, 0, stream>>>(
            rows, (const uint4*)o, (const uint4*)dout, delta, lse, inv, (uint4*)aug_lse,
            (uint4*)aug_delta, (float4*)dq_acc);
    else
        bwd_preprocess_kernel<64><<<(int)blocks, 256, 0, stream>>>(
            rows, (const uint4*)o, (const uint4*)dout, delta, lse, inv, (uint4*)aug_lse,
            (uint4*)aug_delta, (float4*)dq_acc);
    return cudaGetLastError();
}

// fp32 -> bf16, 8 elements per thread step.
__global__ void __launch_bounds__(256) f32_to_bf16_kernel(int64_t n8, const float4* __restrict__ in,
                                                          uint4* __restrict__ out)
{
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8;
         i += (int64_t)gridDim.x * blockDim.x) {
        const float4 a = __ldg(in + 2 * i);
        const float4 b = __ldg(in + 2 * i + 1);
        out[i] = make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(b.x, b.y),
                            pack_bf16x2(b.z, b.w));
    }
}

cudaError_t launch_f32_to_bf16(int64_t n, const float* in, void* out, int num_sms,
                               cudaStream_t stream)
{
    const int64_t n8 = n / 8;
    int64_t blocks = (n8 + 255) / 256;
    const int64_t cap = (int64_t)num_sms * 8;
    if (blocks > cap)
        blocks = cap;
    if (blocks < 1)
        blocks = 1;
    f32_to_bf16_kernel<<<(int)blocks, 256, 0, stream>>>(n8, (const float4*)in, (uint4*)out);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Bounded-wait self-test: every thread waits on a barrier that nothing will
// complete; the wait gives up after limit_ns and records the timeout.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(64) selftest_timeout_kernel(DevStatus* status, uint64_t limit_ns)
{
    __shared__ uint64_t bar;
    __shared__ uint32_t abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0u;
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    WaitCtx w{&abort_flag, status, limit_ns};
    mbar_wait(&bar, 0, w, 99);
    __syncthreads();
}

cudaError_t launch_selftest_timeout(DevStatus* status, uint64_t limit_ns, cudaStream_t stream)
{
    selftest_timeout_kernel<<<1, 64, 0, stream>>>(status, limit_ns);
    return cudaGetLastError();
}

}  // namespace dfa
