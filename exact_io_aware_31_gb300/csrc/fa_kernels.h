// Internal launch interface between the C ABI (fa_api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>

#include "fa_dropout.cuh"

namespace fa {

struct FwdLaunch {
  const CUtensorMap* tm_q;
  const CUtensorMap* tm_k;
  const CUtensorMap* tm_v;
  const CUtensorMap* tm_o;  // bf16 [BH, N, d] output, 64-column x 32-row boxes (stored with TMA at d = 64)
  void* o;
  float* lse;
  int BH, N, d;
  int causal;
  float c2;  // scale * log2(e)
  int* status;
  int grid;
  int dropout = 0;  // 1: dropout on the probabilities with `drop`
  DropParams drop;
  int fp8 = 0;      // 1: tm_q, tm_k are E4M3 codes (d = 128); c2 includes their descale factors
};

struct BwdLaunch {
  const CUtensorMap* tm_q;
  const CUtensorMap* tm_k;
  const CUtensorMap* tm_v;
  const CUtensorMap* tm_do;
  const CUtensorMap* tm_dqacc;  // fp32 [BH, N, d] accumulator, 32-column boxes (d = 64 path)
  const CUtensorMap* tm_dk;     // bf16 [BH, N, d] outputs, 64-column boxes (stored with TMA at d = 64)
  const CUtensorMap* tm_dv;
  const void* o;
  const void* dout;
  const float* lse;
  void* dq;
  void* dk;
  void* dv;
  float* dq_acc;  // [BH, N, d] fp32
  float* lse2;    // [BH, Npad] lse * log2(e), +inf past N
  float* dsum;    // [BH, Npad] D = rowsum(dO * O), 0 past N
  int BH, N, Npad, d;
  int causal;
  float scale;
  float c2;
  int* status;
  int grid;
  int pre_grid;
  int with_dq = 1;  // 0: deterministic backward (dK/dV kernel without dQ, dQ from fa_bwd_dq)
  int dq_grid = 0;
  int dropout = 0;  // 1: gradients of the forward with dropout `drop`
  DropParams drop;
};

// Split-KV forward (decode): Nq <= 8 queries per head against Nk keys.
struct DecLaunch {
  const CUtensorMap* tm_q;  // [BH, Nq, d] bf16, 64-column x 128-row boxes (rows past Nq read as zero)
  const CUtensorMap* tm_k;  // [BH, Nk, d] bf16, 64-column x 128-row boxes
  const CUtensorMap* tm_v;
  const void* q;            // [BH, Nq, d] bf16
  void* o;                  // [BH, Nq, d] bf16
  float* lse;               // [BH, Nq] fp32, natural log
  float* part_o;            // [splits, BH, Nq, d] fp32 partial outputs (splits > 1)
  float* part_lse2;         // [splits, BH, Nq] fp32 partial logsumexp, base 2 (splits > 1)
  int BH, Nq, Nk, d;
  int causal;
  int splits;
  int cluster;  // 1: the splits of a head run as one cluster and merge in shared memory
  float c2;  // scale * log2(e)
  int* status;
};

cudaError_t launch_fwd(const FwdLaunch& a, cudaStream_t stream);
cudaError_t launch_decode(const DecLaunch& a, cudaStream_t stream);
// Queries from which the split-KV forward runs its contractions on the tensor
// cores (fewer run on the CUDA cores).
constexpr int kDecodeMmaMinNq = 3;
// Clusters of `cluster` decode split CTAs that can be resident at once (0: none).
int decode_max_clusters(int d, int nq, int causal, int cluster);
cudaError_t launch_bwd_pre(const BwdLaunch& a, cudaStream_t stream);
cudaError_t launch_bwd_main(const BwdLaunch& a, cudaStream_t stream);
cudaError_t launch_bwd_conv(const BwdLaunch& a, cudaStream_t stream);
cudaError_t launch_bwd_dq(const BwdLaunch& a, cudaStream_t stream);
int bwd_dq_units(int BH, int N);
int fwd_units(int BH, int N);
int bwd_units(int BH, int N);

}  // namespace fa
