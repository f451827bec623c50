// verify.cuh -- argument blocks of the verify kernels (internal).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace mtp {

constexpr int kCandCap = 4096;     // candidates kept per row by the sampling verifier
constexpr int kScanChunk = 32768;  // tokens per (row, chunk) work item of its scans

struct VerifyGreedyArgs {
    const void* logits;
    int B, N;
    long long V;
    const int32_t* drafts;
    int32_t* out_tokens;
    int32_t* out_n_accept;
    WsHeader* hdr;
    unsigned long long* amax;  // [B * (1+N)], zeroed before the launch
};

struct VerifySampleArgs {
    const void* tgt;
    const void* dft;
    int bf16;
    int B, N;
    long long V;
    const int32_t* drafts;
    const int32_t* hist;
    int H;
    int hist_stride;             // row stride of hist (>= H)
    float temp, top_p, min_p, rep, pres;
    unsigned long long seed, offset;
    int32_t* out_tokens;
    int32_t* out_n_accept;
    WsHeader* hdr;
    unsigned long long* rowmax;  // [rows], zeroed before the launch
    unsigned int* cand_cnt;      // [rows], zeroed before the launch
    int32_t* n_keep;             // [rows]
    float* w_keep;               // [rows]
    int32_t* cand_id;            // [rows, kCandCap]
    float* cand_w;               // [rows, kCandCap]
    float* resid;                // [B, kCandCap]
    unsigned long long timeout_ns;
    int draft_k;                 // >= 0: draft sampling, row b = sequence b's logits at draft step draft_k
};

cudaError_t launch_verify_greedy(const VerifyGreedyArgs& a, int ldtype, int num_sms, cudaStream_t s);
cudaError_t launch_verify_sample(const VerifySampleArgs& a, int grid, cudaStream_t s);
int verify_sample_max_grid(int num_sms);

}  // namespace mtp
