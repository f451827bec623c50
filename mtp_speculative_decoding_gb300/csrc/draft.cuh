// draft.cuh -- argument block of the persistent draft-block kernel (internal).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace mtp {

// keys per staged attention sub-chunk: 64, or 32 for rows above 512 bytes
__host__ __device__ constexpr int attn_keys(int hd, int wbytes) { return hd * wbytes <= 512 ? 64 : 32; }
constexpr int kAttnPad = 16;       // bytes of padding per staged K/V row
constexpr int kMaxGrid = 1024;     // upper bound on CTAs of the persistent grid

struct KView {
    const void* k;
    const void* v;
    long long sb, sh, st;
    int cap, window;
    float theta;
    int pad_;
};

struct BlkW {
    const void *w_q, *w_o, *w_gate, *w_up, *w_down;
    const float *attn_norm, *q_norm, *post_attn_norm, *pre_ffn_norm, *post_ffn_norm;
    int view;
    int pad_;
};

struct DraftParams {
    int d_t, d_a, L, Hq, hd, Hkv, F, V, B, N;
    float eps, attn_scale, emb_scale, softcap;
    const void* tok_embd;
    const float* norm_e;
    const float* norm_h;
    const void* w_pre;
    const float* final_norm;
    const void* w_post;
    BlkW blk[MTP_MAX_BLOCKS];
    KView views[MTP_MAX_VIEWS];
    const int32_t* kv_len;
    const int32_t* last_tok;
    const float* h_prev;
    int32_t* out_drafts;
    float* out_h_last;
    float* out_logits;
    // workspace
    WsHeader* hdr;
    unsigned int* att_cnt;       // [B * Hkv] last-arriver counters (self-resetting)
    unsigned long long* amax;    // [N * B] packed argmax keys
    float *XB, *XM, *QR, *OB, *YB, *MB, *Y2, *HN;
    float* PART;                 // attention partials
    float* ACT;                  // [B, kmax] staged activations (global mode)
    int act_smem;                // 1: activations staged per CTA in shared memory
    int kmax;
    unsigned long long timeout_ns;
};

cudaError_t launch_draft_f32(const DraftParams& p, int grid, size_t smem, cudaStream_t s);
cudaError_t launch_draft_bf16(const DraftParams& p, int grid, size_t smem, cudaStream_t s);
int draft_blocks_per_sm_f32(int hd, size_t smem);
int draft_blocks_per_sm_bf16(int hd, size_t smem);

cudaError_t launch_barrier_timeout_probe(WsHeader* hdr, unsigned long long limit_ns, cudaStream_t s);

}  // namespace mtp
