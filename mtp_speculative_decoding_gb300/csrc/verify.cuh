// verify.cuh -- argument blocks and launchers of the verify and sampling
// kernels (internal).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "sample.cuh"

namespace mtp {

struct VerifyGreedyArgs {
    const void* logits;
    int B, N;
    long long V;
    const int32_t* drafts;
    int32_t* out_tokens;
    int32_t* out_n_accept;
    WsHeader* hdr;
    unsigned long long* amax;  // [B * (1+N)], zeroed before the launch
    int split;                 // V-chunks per row (set by the launcher)
};

cudaError_t launch_verify_greedy(const VerifyGreedyArgs& a, int ldtype, int num_sms, cudaStream_t s);

// Pieces per row and tokens per piece of a sampling launch over `rows` rows
// of V tokens on a grid of about `grid` CTAs.
void sample_piece_plan(long long V, long long rows, int grid, int* ppr, int* piece_len);
// One launch of the sampling kernel over every piece of j (mode 0 or 1): a
// persistent grid of at most the CTAs resident on `sms` SMs.
cudaError_t launch_sample(const SampleJob& j, int sms, cudaStream_t s);
// CTAs of the sampling kernel resident per SM
int sample_blocks_per_sm();

}  // namespace mtp
