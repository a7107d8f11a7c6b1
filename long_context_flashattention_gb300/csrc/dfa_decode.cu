// dfa_decode.cu -- split-KV decoding: few query tokens against a long K/V
// cache (FlashAttention glossary entry: the Flash-Decoding variant splits the
// keys so that every SM has work, computes one partial per split and merges
// them; the merge is the same LSE rescaling as dfa_lse_merge, Striped
// Attention Guide, "Incremental Online Softmax Rescaling").
//
// HBM-bound: every K/V row is read once and meets only the R = G*T query rows
// of its head (G = Hq/Hkv), a few FLOP per byte, so the products run on the
// CUDA cores, not the tensor core.  One warp per split of split_len keys,
// registers only: lane l owns feature columns [l*C, l*C + C), C = d/32, of
// the R query rows (pre-scaled by scale*log2 e) and of their output rows.
// Per key: C-wide partial dots, a butterfly shuffle sum (every lane gets the
// score), the online softmax update (rescale only when the running max
// grows), O += p v.  Keys are read 8 at a time (coalesced: a warp reads a
// whole 128- or 256-byte row) so several rows are in flight per warp.
// Output: the split's normalised partial (fp32) and LSE; a row that sees no
// key of the split gives (0, -inf), which the merge ignores.
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "dfa_params.h"
#include "dfa_ptx.cuh"

namespace dfa {

namespace dec {

constexpr int kWarps = 4;     // warps (splits) per CTA
constexpr int kMaxRows = 16;  // G * T query rows per kv head
constexpr int kUnroll = 8;    // keys loaded ahead

template <int C>
struct Vec;
template <>
struct Vec<4> {
    using T = uint2;
    static __device__ __forceinline__ void unpack(const T& x, float* f)
    {
        f[0] = bf16lo(x.x);
        f[1] = bf16hi(x.x);
        f[2] = bf16lo(x.y);
        f[3] = bf16hi(x.y);
    }
};
template <>
struct Vec<2> {
    using T = uint32_t;
    static __device__ __forceinline__ void unpack(const T& x, float* f)
    {
        f[0] = bf16lo(x);
        f[1] = bf16hi(x);
    }
};

template <int D, int R>
__global__ void __launch_bounds__(kWarps * 32) decode_split_kernel(const __grid_constant__ DecodeParams p)
{
    constexpr int C = D / 32;
    using V = Vec<C>;
    const int lane = threadIdx.x & 31;
    const int split = blockIdx.x * kWarps + (threadIdx.x >> 5);
    const int bh = blockIdx.y;  // b * Hkv + hk
    const int b = bh / p.Hkv, hk = bh % p.Hkv;
    const int nsplit = (p.L + p.split_len - 1) / p.split_len;
    if (split >= nsplit)
        return;
    const int Rv = p.G * p.T;  // valid rows (<= R)
    const int64_t k0 = (int64_t)split * p.split_len;
    const int64_t k1 = min((int64_t)p.L, k0 + p.split_len);
    const typename V::T* kb =
        reinterpret_cast<const typename V::T*>((const __nv_bfloat16*)p.k + (size_t)bh * p.L * D) +
        lane;
    const typename V::T* vb =
        reinterpret_cast<const typename V::T*>((const __nv_bfloat16*)p.v + (size_t)bh * p.L * D) +
        lane;
    float q[R][C], o[R][C], m[R], l[R];
    int64_t lim[R];  // last visible key position of each row
#pragma unroll
    for (int r = 0; r < R; ++r) {
        m[r] = -INFINITY;
        l[r] = 0.f;
        const int g = r / p.T, tq = r - g * p.T;
        const bool valid = r < Rv;
        const size_t qrow = ((size_t)b * p.Hq + hk * p.G + (valid ? g : 0)) * p.T + (valid ? tq : 0);
        const typename V::T qv = reinterpret_cast<const typename V::T*>(
            (const __nv_bfloat16*)p.q + qrow * D)[lane];
        float f[C];
        V::unpack(qv, f);
#pragma unroll
        for (int c = 0; c < C; ++c) {
            q[r][c] = f[c] * p.scale_log2;
            o[r][c] = 0.f;
        }
        lim[r] = !valid ? -1 : (p.causal ? p.q_pos0 + tq : (int64_t)p.L - 1);
    }
    for (int64_t j0 = k0; j0 < k1; j0 += kUnroll) {
        typename V::T kr[kUnroll], vr[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t j = min(j0 + u, k1 - 1);
            kr[u] = __ldg(kb + (size_t)j * (D / C));
            vr[u] = __ldg(vb + (size_t)j * (D / C));
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t j = j0 + u;
            float kf[C], vf[C];
            V::unpack(kr[u], kf);
            V::unpack(vr[u], vf);
#pragma unroll
            for (int r = 0; r < R; ++r) {
                float s = 0.f;
#pragma unroll
                for (int c = 0; c < C; ++c)
                    s = fmaf(q[r][c], kf[c], s);
#pragma unroll
                for (int off = 16; off > 0; off >>= 1)
                    s += __shfl_xor_sync(0xffffffffu, s, off);
                if (j < k1 && j <= lim[r]) {
                    if (s > m[r]) {
                        const float a = exp2f(m[r] - s);  // 0 for the first key
                        l[r] *= a;
#pragma unroll
                        for (int c = 0; c < C; ++c)
                            o[r][c] *= a;
                        m[r] = s;
                    }
                    const float pj = exp2f(s - m[r]);
                    l[r] += pj;
#pragma unroll
                    for (int c = 0; c < C; ++c)
                        o[r][c] = fmaf(pj, vf[c], o[r][c]);
                }
            }
        }
    }
    const size_t rows = (size_t)p.B * p.Hq * p.T;
    float* o_part = p.o_part + (size_t)split * rows * D;
    float* lse_part = p.lse_part + (size_t)split * rows;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        if (r >= Rv)
            continue;
        const int g = r / p.T, tq = r - g * p.T;
        const size_t orow = ((size_t)b * p.Hq + hk * p.G + g) * p.T + tq;
        const float inv = l[r] > 0.f ? 1.f / l[r] : 0.f;
#pragma unroll
        for (int c = 0; c < C; ++c)
            o_part[orow * D + lane * C + c] = o[r][c] * inv;
        if (lane == 0)
            lse_part[orow] =
                l[r] > 0.f ? (m[r] + log2f(l[r])) * 0.69314718055994531f : -INFINITY;
    }
}

template <int D, int R>
cudaError_t launch(const DecodeParams& p, int splits, cudaStream_t stream)
{
    const dim3 grid((splits + kWarps - 1) / kWarps, p.B * p.Hkv);
    decode_split_kernel<D, R><<<grid, kWarps * 32, 0, stream>>>(p);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_rows(const DecodeParams& p, int splits, cudaStream_t stream)
{
    const int R = p.G * p.T;
    if (R <= 1)
        return launch<D, 1>(p, splits, stream);
    if (R <= 2)
        return launch<D, 2>(p, splits, stream);
    if (R <= 4)
        return launch<D, 4>(p, splits, stream);
    if (R <= 8)
        return launch<D, 8>(p, splits, stream);
    return launch<D, 16>(p, splits, stream);
}

}  // namespace dec

cudaError_t launch_decode_split(int d, const DecodeParams& p, int splits, cudaStream_t stream)
{
    return d == 128 ? dec::launch_rows<128>(p, splits, stream)
                    : dec::launch_rows<64>(p, splits, stream);
}

int decode_max_rows() { return dec::kMaxRows; }

}  // namespace dfa
