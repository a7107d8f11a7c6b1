// dfa_launch.h -- host-side launch entry points of the kernels (internal).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "dfa_params.h"

namespace dfa {

struct DevStatus;
struct PermuteParams;

cudaError_t launch_attn_fwd(int d, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const FwdParams& p, int grid,
                            cudaStream_t stream);
int fwd_rows_per_unit();

cudaError_t launch_attn_bwd(int d, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& tdo,
                            const CUtensorMap& tal, const CUtensorMap& tad, const BwdParams& p,
                            int grid, cudaStream_t stream);
int bwd_rows_per_unit();
int bwd_query_rows_per_step();

cudaError_t launch_lse_merge(int64_t rows, int d, int k, const float* o_parts,
                             const float* lse_parts, void* o_out, float* lse_out, int out_fp32,
                             int accumulate, int num_sms, cudaStream_t stream);
cudaError_t launch_permute(const PermuteParams& pp, const void* in, void* out, int vec_bytes,
                           int num_sms, cudaStream_t stream);
cudaError_t launch_decode_split(int d, const DecodeParams& p, int splits, cudaStream_t stream);
int decode_max_rows();
struct RopeParams;
cudaError_t launch_permute_rope(const RopeParams& rp, const void* in, void* out, int num_sms,
                                cudaStream_t stream);
// Per query row of the backward: the 32-byte K-slice records of -LSE/scale
// and -D (D = dO . O computed here from o and dout, or read from delta when
// o is NULL), and, if dq_acc is not NULL, zeroing of its dQ accumulator row.
cudaError_t launch_bwd_preprocess(int64_t rows, int d, const void* o, const void* dout,
                                  const float* delta, const float* lse, float scale,
                                  void* aug_lse, void* aug_delta, float* dq_acc, int num_sms,
                                  cudaStream_t stream);
constexpr int kAugRowBytes = 32;  // one record: 16 bf16
cudaError_t launch_f32_to_bf16(int64_t n, const float* in, void* out, int num_sms,
                               cudaStream_t stream);
cudaError_t launch_selftest_timeout(DevStatus* status, uint64_t limit_ns, cudaStream_t stream);

}  // namespace dfa
