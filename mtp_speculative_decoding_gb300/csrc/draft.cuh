// draft.cuh -- argument block of the persistent draft-block kernel (internal).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace mtp {

constexpr int kMaxGrid = 1024;     // upper bound on CTAs of the persistent grid

// phases of one draft step
enum Phase { PH_PRE, PH_Q, PH_O, PH_FFN1, PH_FFN2, PH_POST, PH_HEAD };

// Shape of the attention phase for head dimension hd and element size wb.
// A K or V row is split over LPR lanes, CPL 16-byte chunks each; a warp
// reads KPW rows side by side and stages R keys (K and V rows, 4 KB) per
// round in each of kAttnStages ring slots; HG query heads share a pass.
struct AttnGeom {
    int RB, CPR, LPR, CPL, KPW, EPC, DPL, R, RL, SB, HG;
};
__host__ __device__ constexpr AttnGeom attn_geom(int hd, int wb) {
    const int RB = hd * wb, CPR = RB / 16, LPR = CPR < 32 ? CPR : 32, CPL = CPR / LPR, KPW = 32 / LPR;
    const int EPC = 16 / wb, DPL = CPL * EPC, R = 2048 / RB > KPW ? 2048 / RB : KPW;
    const int HG = 32 / DPL >= 4 ? 4 : (32 / DPL >= 1 ? 32 / DPL : 1);
    return AttnGeom{RB, CPR, LPR, CPL, KPW, EPC, DPL, R, R / KPW, 2 * R * RB, HG};
}
constexpr int kAttnStages = 2;     // single-sequence kernel
constexpr int kAttnStagesTc = 3;   // batched (tensor-core) kernel: 3 measured 6% faster per launch than 2 at B = 64
// LM head of one sequence: four groups of four warps, each with kHeadSlots
// one-row slots; rows of up to kHeadMaxChunks 16-byte chunks
constexpr int kHeadGroups = 4;
constexpr int kHeadSlots = 3;
constexpr int kHeadMaxChunks = 640;
// Batched projections on tensor cores (bf16 weights, B >= kTcMinBatch):
// 128-row weight tiles, K steps of 64, a tc_stages-deep operand ring.  From
// two sequences the tensor-core head beats the CUDA-core GEMV over B columns
// (measured, draft launch at the Gemma shape: B = 2 3.29 -> 2.22 ms, B = 4
// 4.96 -> 2.60, B = 6 10.8 -> 2.47); one sequence keeps the bulk-copy head.
constexpr int kTcMinBatch = 2;
constexpr int kTcTileM = 128;
constexpr int kTcTileK = 64;
constexpr int kTcMaxStages = 8;
constexpr size_t kTcSmemBudget = 128 * 1024;
// LM head on tensor cores: the batch (rows >= B zero) is the MMA's M = 64
// side and 256 rows of the token table its N side, so each MMA takes 8 KB of
// the table; stages of one 64 x 256 table box and the batch's 64 x 64 block(s)
constexpr int kTcHeadM = 64;
constexpr int kTcHeadN = 256;
constexpr size_t kTcHeadSmemBudget = 200 * 1024;
constexpr int kTcHeadCols = 512;   // tensor-memory columns: two 256-column accumulators
// Projection epilogue staging after the operand ring: a 128-row output tile
// as fp32 [b][128] (512 bytes per sequence), then (post-projection) the
// tile's two 64-column blocks of h's bf16 high and low parts in the head
// operand's swizzled layout
constexpr size_t kTcStageBytes = (size_t)kTcHeadM * kTcTileM * 4 + 2 * 2 * (size_t)kTcHeadM * 128;

// floats per attention partial: o[grp][hd], m[grp], l[grp], padded to 16 bytes
__host__ __device__ constexpr int attn_psz(int grp, int hd) { return (grp * (hd + 2) + 3) & ~3; }
// float offsets from the rotated queries: warps' (m, l) at grp * hd, merge
// weights and maxima after them, then (16-byte aligned) the per-warp round
// probabilities and rescales
__host__ __device__ constexpr int attn_pb_off(int grp, int hd, int hg) { return (grp * hd + 3 * kWarps * hg + hg + 3) & ~3; }
// dynamic shared memory of the attention phase: the rings, then the above
__host__ __device__ constexpr size_t attn_smem(int hd, int wb, int grp, int nst) {
    return (size_t)kWarps * nst * attn_geom(hd, wb).SB +
           ((size_t)attn_pb_off(grp, hd, attn_geom(hd, wb).HG) +
            (size_t)kWarps * ((attn_geom(hd, wb).RL * attn_geom(hd, wb).HG + attn_geom(hd, wb).HG + 3) & ~3)) *
               sizeof(float);
}

struct KView {
    const void* k;
    const void* v;
    long long sb, sh, st;
    int cap, window;
    float theta;
    int sink;                 // attention-sink positions read with a window (0: none)
    unsigned int cap_magic;   // floor(2^32 / cap): slot = position mod cap by a multiply-high
    unsigned int ring_magic;  // floor(2^32 / (cap - sink)) for the ring above the sink
};

struct BlkW {
    const void *w_q, *w_o, *w_gate, *w_up, *w_down;
    const uint16_t *s_q, *s_o, *s_gate, *s_up, *s_down;   // Q8_0 block scales (binary16) or null
    const float *attn_norm, *q_norm, *post_attn_norm, *pre_ffn_norm, *post_ffn_norm;
    const float* k_norm;   // NextN: the key norm (null for the assistant)
    int view;
    int pad_;
};

struct DraftParams {
    // tensor-core weights, box 64 x 128 with 128-byte swizzle: the token
    // table [V, d_t], then the projections: pre, post, per block q, o, gate,
    // up, down
    CUtensorMap tm_embd;
    CUtensorMap tm_w[2 + 5 * MTP_MAX_BLOCKS];
    int d_t, d_a, L, Hq, hd, Hkv, F, V, B, N;
    float eps, attn_scale, emb_scale, softcap;
    const void* tok_embd;
    const float* norm_e;
    const float* norm_h;
    const void* w_pre;
    const float* final_norm;
    const void* w_post;
    const uint16_t *s_pre, *s_post;   // Q8_0 block scales (binary16) or null
    BlkW blk[MTP_MAX_BLOCKS];
    KView views[MTP_MAX_VIEWS];
    const int32_t* kv_len;
    const int32_t* last_tok;
    const float* h_prev;
    int32_t* out_drafts;
    float* out_h_last;
    float* out_logits;
    float* out_conf;             // [B, N] per-step top-1 softmax probability, or null
    // workspace
    WsHeader* hdr;
    unsigned int* att_cnt;       // [B * Hkv] last-arriver counters (self-resetting)
    unsigned long long* amax;    // [N * B] packed argmax keys
    float *XB, *XM, *QR, *OB, *YB, *MB, *Y2, *HN;
    float* PART;                 // attention partials
    float2* CONF;                // [grid][B] per-CTA softmax-denominator partials (max, sum) of the step's logits
    double* ROPE;                // [MTP_MAX_VIEWS][hd / 2] RoPE inverse frequencies (written at kernel start)
    float2* ROPEQ;               // [B][MTP_MAX_VIEWS][hd / 2] (cos, sin) at the step's query position
    float* ACT;                  // [B, kmax] staged activations (global mode)
    int act_smem;                // 1: activations staged per CTA in shared memory
    int head_slotb;              // > 0: one sequence, LM head rows through bulk-copy slots of this many bytes
    int tc_head;                 // 1: LM head on tensor cores
    int Bp, tc_stages, tc_cols;  // batch padded to 16; operand ring depth; tensor-memory columns
    int th_stages;               // LM head ring depth
    uint16_t *XH, *XL;           // bf16 high / low parts of h as the head's tiled operand (kTcHeadM rows, >= B zero)
    int tc_proj;                 // 1: projections on tensor cores (activations staged in global memory)
    int att_fold;                // 1: split attention segments are merged by the O prologue (tc_proj only)
    int sk[6];                   // split-K factor of each projection phase (PH_PRE .. PH_POST)
    uint16_t *XA, *XAL;          // bf16 high / low parts of the current phase input, tiled
    float* PB;                   // [S][B][R] split partials of the last projection (FFN1: R = 2 F)
    int kmax;
    unsigned long long timeout_ns;
    // sampled drafting (temperature > 0): sample_dist parameters, the
    // Philox stream, the penalty history [B, H], the step's logits [B, V]
    // and the sampler's per-row state (zero at launch; see sample.cuh)
    int sampling;
    float s_temp, s_top_p, s_min_p, s_rep, s_pres;
    unsigned long long seed, offset;
    const int32_t* hist;
    int H;
    float* ZB;
    unsigned int* S_row;         // [4][B]: row maximum key, survivor count, overflow flag, pieces done
    int2* S_buf;                 // [B][S_rcap] survivors
    int S_rcap, S_plen, S_ppr;   // survivor capacity per row, tokens per piece, pieces per row
    // centroid-routed LM head (n_cent > 0): centroids [n_cent, d_t] (weight
    // type), token ordering [V] int32, the step's centroid logits [B, n_cent]
    int n_cent, cent_k;
    const void* cent;
    const int32_t* cord;
    float* CL;
    // dense NextN drafter (nextn = 1): one block with a fused query / key /
    // value projection into QR, its own KV (views[0], written by the kernel),
    // catch-up rows before the draft steps, the block output as the chain
    int QS;                      // floats per sequence in QR: Hq hd, or (Hq + 2 Hkv) hd for NextN
    int nextn;
    int M;                       // catch-up rows per sequence at most
    const int32_t* n_cu;         // [B] catch-up rows of each sequence, or null (none)
    const int32_t* cu_tok;       // [B, M] their tokens
    const float* cu_h;           // [B, M, d_t] the hidden states paired with them
    float* HX;                   // [B, d_t] the block output: the next step's hidden state
};

cudaError_t launch_draft_f32(const DraftParams& p, int grid, size_t smem, cudaStream_t s);
cudaError_t launch_draft_bf16_cc(const DraftParams& p, int grid, size_t smem, cudaStream_t s);
cudaError_t launch_draft_bf16_tc(const DraftParams& p, int grid, size_t smem, cudaStream_t s);
// bf16 table and KV, Q8_0 projections (CUDA-core paths); head_dim 64, 128 or 256
cudaError_t launch_draft_q8(const DraftParams& p, int grid, size_t smem, cudaStream_t s);
int draft_blocks_per_sm_q8(int hd, size_t smem);
// bf16 table and KV, Q4_0 projections (CUDA-core paths); head_dim 64, 128 or 256
cudaError_t launch_draft_q4(const DraftParams& p, int grid, size_t smem, cudaStream_t s);
int draft_blocks_per_sm_q4(int hd, size_t smem);
int draft_blocks_per_sm_f32(int hd, size_t smem);
int draft_blocks_per_sm_bf16_cc(int hd, size_t smem);
int draft_blocks_per_sm_bf16_tc(int hd, size_t smem);

cudaError_t launch_barrier_timeout_probe(WsHeader* hdr, unsigned long long limit_ns, cudaStream_t s);

}  // namespace mtp
