/*
 * mtp.h -- C ABI of the GB300 MTP speculative-decoding hot path.
 *
 * Five operations, all asynchronous on a caller-supplied CUDA stream:
 *
 *   mtp_draft_block    N chained draft steps of an MTP assistant head that
 *                      cross-attends into the target's KV cache, in ONE
 *                      persistent launch (token -> embedding -> hidden-state
 *                      chain stays on the device between steps).
 *   mtp_verify_greedy  longest greedy-matching prefix + bonus token from the
 *                      target's (1+N) x V verify logits.
 *   mtp_verify_sample  exact speculative sampling at temp > 0.
 *   mtp_sample_drafts  the draws of a sampling drafter from given draft
 *                      logits (the q the sampling verifier checks against).
 *   mtp_nextn_draft    the dense NextN self-speculation drafter: its own
 *                      block and its own KV, the catch-up on the accepted
 *                      rows, then N chained draft steps, in ONE launch.
 *
 * Definitions are those of the pages this library implements:
 *   [G4] "Gemma 4 MTP -- Multi-Token Prediction speculative decoding":
 *        sec. 4 "Per-step MTP graph" (the draft step), sec. 5 "KV sharing"
 *        (read-only cross-attention, one mask for all steps), sec. 6 (the
 *        public API this one replaces: llama_decode_mtp_async / _wait).
 *   [NX] "MTP decoding (--mtp)": "Requirements" (enorm / hnorm / eh_proj) and
 *        "How it is wired" (greedy longest-prefix accept + bonus token).
 *   [FN] "Fused NextN draft graph": one launch + one readback for N steps;
 *        delta 6 (frozen-prefix cross-attention).
 *   [SP] "opus-mtp-turbo: Track 1 report", item 4 (exact temp > 0
 *        verification: sample_dist, accept with p/q, residual max(p - q, 0)).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every pointer argument is DEVICE memory owned by the caller, unless its
 *   comment says "host".  The library never allocates, frees or copies
 *   buffers of its own, never synchronizes the stream (except
 *   mtp_last_error, which says so) and keeps no state between calls.
 * - Scratch space is the caller's workspace `ws` (`ws_bytes` bytes, 256-byte
 *   aligned, device memory), sized by mtp_workspace_size().  Calls that share
 *   a workspace must be ordered on one stream.
 * - Return value: MTP_OK, or a negative MTP_ERR_* code when the arguments are
 *   rejected on the host (nothing is launched then) or a launch fails.
 *   Errors found while the kernels run (a grid barrier that timed out, a
 *   candidate set that overflowed) are written to a status word inside the
 *   workspace and read back with mtp_last_error().
 * - Row-major layouts; every row start must be 16-byte aligned (row lengths
 *   in elements: multiples of 8 for bf16, 4 for fp32).
 */
#ifndef MTP_H
#define MTP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* a cudaStream_t; NULL is the legacy default stream */
typedef struct CUstream_st *mtp_stream_t;

enum {
    MTP_OK = 0,
    MTP_ERR_ARG = -1,          /* a pointer, size or layout argument is invalid */
    MTP_ERR_UNSUPPORTED = -2,  /* valid, but outside what the kernels implement */
    MTP_ERR_WORKSPACE = -3,    /* ws is NULL, misaligned or smaller than required */
    MTP_ERR_CUDA = -4,         /* a CUDA launch failed */
    MTP_ERR_TIMEOUT = -5,      /* (device status) a grid barrier gave up waiting */
    MTP_ERR_CAPACITY = -6      /* (device status) a sampling candidate set overflowed */
};

enum { MTP_DTYPE_F32 = 0, MTP_DTYPE_BF16 = 1 };
/* projection weight formats (mtp_config.wquant) */
enum { MTP_WQ_NONE = 0, MTP_WQ_Q8_0 = 1, MTP_WQ_Q4_0 = 2 };

#define MTP_MAX_BLOCKS 8
#define MTP_MAX_VIEWS 4
#define MTP_MAX_BATCH 64            /* sequences of one mtp_draft_block call */
#define MTP_MAX_VERIFY_BATCH 65536  /* sequences of one verify or draw call */
#define MTP_MAX_CENTROIDS 8192      /* centroids of a centroid-routed LM head */
#define MTP_MAX_CATCHUP 16          /* catch-up rows per sequence of one mtp_nextn_draft call */

/* Sizes and scalars of the assistant head ([G4] sec. 3-4).
 *   d_t        backbone (target) width: token embedding, h_prev, LM head input
 *   d_a        assistant width
 *   n_blocks   assistant blocks (<= MTP_MAX_BLOCKS)
 *   n_q_heads, head_dim, n_kv_heads   query heads, their width, KV heads of the
 *              target layers cross-attended (n_q_heads % n_kv_heads == 0)
 *   d_ff       GeGLU hidden width
 *   vocab      rows of the tied token-embedding table
 *   wdtype     MTP_DTYPE_BF16 or MTP_DTYPE_F32: weight matrices and KV
 *   rms_eps    RMSNorm epsilon; attn_scale softmax scale, 0 = the default
 *              1/sqrt(head_dim) (rounded to fp32);
 *   emb_scale  token-embedding scale, 0 = the default sqrt(d_t) (Gemma's);
 *   logit_softcap  > 0 applies cap * tanh(z / cap) to the logits, 0 = off
 *   n_centroids    0: the dense tied LM head.  > 0: the centroid-routed head
 *                  of ordered-embedding models ([G4] sec. 3 "Centroid /
 *                  ordered-embeddings LM head"), n_centroids <=
 *                  MTP_MAX_CENTROIDS dividing vocab (MTP_ERR_ARG otherwise;
 *                  above the maximum MTP_ERR_UNSUPPORTED)
 *   centroid_top_k centroids whose candidate lists are scored per step,
 *                  1..n_centroids (ignored for the dense head, must be >= 0)
 *   wquant         MTP_WQ_NONE: the projections (w_pre, w_post and every
 *                  block's w_q, w_o, w_gate, w_up, w_down) are in wdtype.
 *                  MTP_WQ_Q8_0 ("opus-mtp-turbo: Track 1 report", item 3):
 *                  they are Q8_0 codes, int8 [out, in], each with its
 *                  block scales, binary16 [out, in / 32] (see
 *                  mtp_quantize_q8_0); requires wdtype MTP_DTYPE_BF16 (the
 *                  table and KV), head_dim 64, 128 or 256, every input
 *                  width a multiple of 32; runs on the CUDA-core paths.
 *                  MTP_WQ_Q4_0 (the same item's Q4_0 column): Q4_0 codes,
 *                  uint8 [out, in / 2] -- per block of 32 weights 16 bytes,
 *                  byte j holding the code of weight j in its low four bits
 *                  and of weight j + 16 in its high four; the weight is
 *                  (code - 8) times the block's binary16 scale [out, in / 32]
 *                  (see mtp_quantize_q4_0); the same requirements as Q8_0 */
typedef struct mtp_config {
    int32_t d_t, d_a, n_blocks, n_q_heads, head_dim, n_kv_heads, d_ff, vocab;
    int32_t wdtype;
    float rms_eps, attn_scale, emb_scale, logit_softcap;
    int32_t n_centroids, centroid_top_k;
    int32_t wquant, pad_;
} mtp_config;

/* One assistant block.  Matrices are row-major [out, in] in `wdtype`; RMSNorm
 * gains are fp32.  kv_view selects which mtp_kv_view the block attends. */
typedef struct mtp_block_weights {
    const void *attn_norm;       /* fp32 [d_a] */
    const void *w_q;             /* [n_q_heads * head_dim, d_a] */
    const void *q_norm;          /* fp32 [head_dim], shared by all heads */
    const void *w_o;             /* [d_a, n_q_heads * head_dim] */
    const void *post_attn_norm;  /* fp32 [d_a] */
    const void *pre_ffn_norm;    /* fp32 [d_a] */
    const void *w_gate;          /* [d_ff, d_a] */
    const void *w_up;            /* [d_ff, d_a] */
    const void *w_down;          /* [d_a, d_ff] */
    const void *post_ffn_norm;   /* fp32 [d_a] */
    int32_t kv_view;
    int32_t pad_;
    /* MTP_WQ_Q8_0 only (NULL otherwise): block scales of w_q, w_o, w_gate, w_up, w_down */
    const uint16_t *w_q_scale, *w_o_scale, *w_gate_scale, *w_up_scale, *w_down_scale;
    /* mtp_nextn_draft only (NULL otherwise): fp32 [head_dim] key norm, shared by all KV heads */
    const void *k_norm;
} mtp_block_weights;

typedef struct mtp_weights {
    const void *tok_embd;    /* [vocab, d_t]: the TARGET's table, also the tied LM head */
    const void *norm_e;      /* fp32 [d_t]: norm of the scaled token embedding */
    const void *norm_h;      /* fp32 [d_t]: norm of h_prev */
    const void *w_pre;       /* [d_a, 2 d_t]: pre-projection of [norm_e(e); norm_h(h)] */
    const void *final_norm;  /* fp32 [d_a] */
    const void *w_post;      /* [d_t, d_a]: post-projection -> next h_prev */
    mtp_block_weights blk[MTP_MAX_BLOCKS];
    /* centroid-routed head only (NULL for the dense head): */
    const void *centroids;           /* [n_centroids, d_t] in wdtype, 16-byte aligned */
    const int32_t *token_ordering;   /* [vocab]: n_centroids consecutive lists of
                                      * vocab / n_centroids token ids, list j the
                                      * candidates of centroid j */
    /* MTP_WQ_Q8_0 only (NULL otherwise): block scales of w_pre and w_post */
    const uint16_t *w_pre_scale, *w_post_scale;
} mtp_weights;

/* A read-only view of one target KV layer ([G4] sec. 5).  K and V share the
 * layout: element (b, kv head g, slot s, d) at b*stride_b + g*stride_h +
 * s*stride_t + d (elements of `wdtype`; d contiguous).  window == 0 reads
 * positions [0, kv_len[b]) (requires kv_len[b] <= cap, sink == 0); window
 * W > 0 reads the last W positions [lo, kv_len[b]), lo = max(0, kv_len[b] - W),
 * plus the attention sink [0, min(sink, lo)) ("opus-mtp-turbo: Track 1
 * report", item 2: the draft attention reads the first `sink` cells and the
 * window).  Storage: position t lives in slot t for t < sink and in slot
 * sink + (t - sink) % (cap - sink) from there on (a ring of `cap` slots when
 * sink == 0); requires W + sink <= cap.  K is stored after RoPE; V is used as
 * stored.  rope_theta is the RoPE base of the target layer type (applied to
 * the drafter's queries). */
typedef struct mtp_kv_view {
    const void *k, *v;
    int64_t stride_b, stride_h, stride_t;
    int32_t cap, window;
    float rope_theta;
    int32_t sink;
} mtp_kv_view;

/* sample_dist settings ([SP] item 4): repetition penalty (z > 0: z / r, else
 * z * r) and presence penalty (z - pres), once per distinct token of the
 * penalty set, then temperature, min-p (keep p >= min_p * p_max), top-p (keep
 * the shortest prefix, by probability desc / id asc, whose mass reaches
 * top_p), renormalising after each cut.  top_k must be 0 (off). */
typedef struct mtp_sample_params {
    float temp, top_p, min_p, rep_penalty, presence_penalty;
    int32_t top_k;
} mtp_sample_params;

/* Q8_0 quantisation of a row-major fp32 matrix [rows, cols] on the host
 * ("opus-mtp-turbo: Track 1 report", item 3, ggml's Q8_0 rule): per block of
 * 32 consecutive weights of a row, d = max |w| / 127 (fp32), stored as
 * binary16 (round to nearest even); codes q = round(w * (1 / d)) in fp32,
 * halves away from zero, 0 when d = 0.  The weight a code stands for is
 * binary16(d) * q.  Host pointers: w [rows, cols], codes [rows, cols] int8,
 * scales [rows, cols / 32].  cols must be a multiple of 32 (MTP_ERR_ARG).
 * Synchronous, no device work. */
int mtp_quantize_q8_0(const float *w, int64_t rows, int64_t cols, int8_t *codes, uint16_t *scales);
/* Q4_0 quantisation on the host ("opus-mtp-turbo: Track 1 report", item 3,
 * the Q4_0 format; the scale by ggml's rule, where the report's quantiser
 * picks it by Lloyd iterations): per block of 32 consecutive weights of a row,
 * m = the weight of largest magnitude (the first on ties), d = m / -8 (fp32),
 * stored as binary16 (round to nearest even); codes q = min(15, trunc(w * (1 /
 * d) + 8.5)) in fp32, 8 when d = 0.  Host pointers: w [rows, cols], codes
 * [rows, cols / 2] uint8 (layout as for MTP_WQ_Q4_0), scales [rows, cols /
 * 32].  cols must be a multiple of 32 (MTP_ERR_ARG).  Synchronous, no device
 * work. */
int mtp_quantize_q4_0(const float *w, int64_t rows, int64_t cols, uint8_t *codes, uint16_t *scales);

/* Workspace bytes needed by any of the operations for these sizes (B
 * sequences, N drafts, vocabulary V).  cfg may be NULL when only the verify
 * and draw calls will use the workspace (then B <= MTP_MAX_VERIFY_BATCH,
 * else B <= MTP_MAX_BATCH).  Returns 0 for invalid sizes. */
size_t mtp_workspace_size(const mtp_config *cfg, int B, int N, int V);

/* N chained draft steps for B sequences ([G4] sec. 4-5, [NX], [FN]).
 * Step k of sequence b consumes token tok_k (last_tok[b] for k = 0, the draft
 * of step k-1 after) and hidden state h_k (h_prev[b] for k = 0, the previous
 * step's post-projection after):
 *   e = tok_embd[tok_k] * emb_scale
 *   x = w_pre [rmsnorm(e; norm_e); rmsnorm(h_k; norm_h)]
 *   per block: q = rope(qnorm(w_q rmsnorm(x)), pos = kv_len[b] + k);
 *              o = GQA softmax cross-attention of q into the block's view;
 *              x += rmsnorm(w_o o); x += rmsnorm(w_down(gelu_tanh(w_gate n) * w_up n)),
 *              n = rmsnorm(x; pre_ffn_norm)
 *   h_{k+1} = w_post rmsnorm(x; final_norm);  z = tok_embd h_{k+1} (softcap)
 *   (centroid-routed head, cfg->n_centroids > 0: z is -1e30 except at the
 *   candidates, the lists of the centroid_top_k centroids with the largest
 *   centroids[j] . h_{k+1} (lower j on ties), where z_t = tok_embd[t] h_{k+1}
 *   (softcap); an ordering entry outside [0, vocab) is skipped and sets the
 *   status word to MTP_ERR_ARG)
 *   draft_k = argmax z (lowest index on ties), or, when sp != NULL and
 *   sp->temp > 0, a draw from sample_dist(z) with penalty set hist[b] u
 *   {draft_0..draft_{k-1}} and the Philox-4x32-10 uniform of counter
 *   (b, 4k + 0, offset lo, offset hi), key (seed lo, seed hi).
 * Arguments:
 *   views[n_views]       KV views (host array of structs; data on device)
 *   kv_len [B] int32     attn_pos + 1 of each sequence, >= 1
 *   last_tok [B] int32   the last accepted token
 *   h_prev [B, d_t] fp32 the target's hidden state at that token
 *   sp                   host pointer or NULL (greedy); with temp > 0 the
 *                        settings are checked as for mtp_verify_sample
 *                        (MTP_ERR_ARG; top_k != 0: MTP_ERR_UNSUPPORTED), and
 *                        a kept set over 4096 candidates sets the status word
 *                        to MTP_ERR_CAPACITY
 *   hist [B, H] int32    penalty history (newest last; entries < 0 ignored);
 *                        used only when sampling; may be NULL when H == 0
 *   out_drafts [B, N] int32
 *   out_h_last [B, d_t] fp32, or NULL: h after the last step
 *   out_logits [B, N, vocab] fp32, or NULL: every step's logits (diagnostic)
 *   out_conf [B, N] fp32, or NULL: each step's confidence, the softmax
 *                        probability of its largest logit, 1 / sum_v
 *                        exp(z_v - max z) over the step's logits (after the
 *                        softcap, NaN left out) -- the draft loop's
 *                        confidence that [NX] "Stopping early when the head
 *                        is unsure" compares with p_min.  The caller trims a
 *                        row's drafts at the first step below its p_min
 *                        before verifying; the drafts themselves do not
 *                        depend on it.
 * B <= MTP_MAX_BATCH, 1 <= N <= 16.  One cooperative launch (plus a 256-byte
 * workspace memset); no host round-trip between steps. */
int mtp_draft_block(const mtp_config *cfg, const mtp_weights *w,
                    const mtp_kv_view *views, int n_views,
                    const int32_t *kv_len, int B, int N,
                    const int32_t *last_tok, const float *h_prev,
                    const mtp_sample_params *sp, uint64_t seed, uint64_t offset,
                    const int32_t *hist, int H,
                    int32_t *out_drafts, float *out_h_last, float *out_logits,
                    float *out_conf, void *ws, size_t ws_bytes, mtp_stream_t stream);

/* The dense NextN drafter ([NX] "Requirements", "How it is wired", "The
 * catch-up runs on the accepted prefix"; [FN] "The two MTP lanes": NextN runs
 * its own block over its own KV).  One block at the backbone width d = d_t.
 * The drafter's KV `dkv` holds kv_len[b] rows of sequence b, the row of
 * position t in slot t (window 0, sink 0, kv_len[b] + n_cu[b] + N <= cap);
 * this call WRITES rows kv_len[b] .. kv_len[b] + n_cu[b] + N - 1 of it.
 * A row consumes a token t at position pos and a hidden state h:
 *   x = w_pre [rmsnorm(tok_embd[t] * emb_scale; norm_e); rmsnorm(h; norm_h)]
 *       (w_pre the eh_proj [d, 2d]; emb_scale 0 = the default 1)
 *   a = rmsnorm(x; attn_norm);  [q; k; v] = w_q a  (w_q [(Hq + 2 Hkv) hd, d]:
 *       query rows, then key rows, then value rows)
 *   per KV head: key = rope(rmsnorm(k_g; k_norm), pos), value = v_g, both
 *       stored at slot pos rounded to wdtype
 * Catch-up rows stop there.  A draft step goes on:
 *   per query head: q_h = rope(rmsnorm(q_h; q_norm), pos) attends (GQA,
 *       scale attn_scale) to the rows [0, pos] of KV head h / (Hq / Hkv)
 *   x += w_o o;  x += w_down(silu(w_gate n) * w_up n), n = rmsnorm(x; pre_ffn_norm)
 *   h' = x (the next step's hidden state);  z = tok_embd rmsnorm(x; final_norm)
 *       (final_norm the shared head's norm; optional softcap); draft = argmax z
 *       (lowest index on ties)
 * Rows of sequence b: catch-up row j < n_cu[b] consumes (cu_tok[b, j],
 * cu_h[b, j]) at position kv_len[b] + j -- the accepted drafts with the
 * target's hidden states at the positions before them; draft step k consumes
 * (last_tok[b], h_prev[b]) for k = 0 -- the bonus token with the target's
 * hidden state before it -- and (draft k-1, h' of step k-1) after, at
 * position kv_len[b] + n_cu[b] + k.  The next call's kv_len is kv_len +
 * n_cu + 1: the rows of steps k >= 1 are the drafter's own guesses, and the
 * next call's catch-up rewrites the accepted ones (no rollback is needed).
 * Arguments:
 *   cfg        d_a == d_t, n_blocks == 1, n_centroids == 0; wquant NONE,
 *              Q8_0 or Q4_0 (then w_pre_scale and blk[0]'s w_q, w_o,
 *              w_gate, w_up, w_down scales are required); rope_theta comes
 *              from dkv
 *   w          tok_embd, norm_e, norm_h, w_pre (eh_proj), final_norm (head
 *              norm); blk[0]: attn_norm, w_q (fused), q_norm, k_norm, w_o,
 *              pre_ffn_norm, w_gate, w_up, w_down (w_post, post_attn_norm,
 *              post_ffn_norm, centroids and w_post_scale unused, may be NULL)
 *   dkv        host pointer to one view (data on device, written)
 *   kv_len [B] int32 >= 0;  n_cu [B] int32 in [0, M] (NULL: all 0)
 *   cu_tok [B, M] int32, cu_h [B, M, d] fp32 (only rows j < n_cu[b] are read;
 *              NULL when M == 0);  0 <= M <= MTP_MAX_CATCHUP
 *   last_tok [B] int32;  h_prev [B, d] fp32
 *   out_drafts [B, N] int32;  out_h_last [B, d] fp32 or NULL: h' of the last
 *              step;  out_logits [B, N, vocab] fp32 or NULL;  out_conf [B, N]
 *              fp32 or NULL (as for mtp_draft_block)
 * Greedy only ([NX]: speculation there requires greedy decoding).  B <=
 * MTP_MAX_BATCH, 1 <= N <= 16.  Host-checked arguments return MTP_ERR_ARG /
 * MTP_ERR_UNSUPPORTED; a kv_len, n_cu or token out of range sets the status
 * word to MTP_ERR_ARG and the kernel returns before writing anything.  One
 * cooperative launch (plus a 256-byte workspace memset). */
int mtp_nextn_draft(const mtp_config *cfg, const mtp_weights *w, const mtp_kv_view *dkv,
                    const int32_t *kv_len, int B, int N,
                    const int32_t *n_cu, const int32_t *cu_tok, const float *cu_h, int M,
                    const int32_t *last_tok, const float *h_prev,
                    int32_t *out_drafts, float *out_h_last, float *out_logits, float *out_conf,
                    void *ws, size_t ws_bytes, mtp_stream_t stream);
/* Greedy verify ([NX] How it is wired).  B <= MTP_MAX_VERIFY_BATCH.  logits [B, 1+N, V] in ldtype (row i
 * is the target's distribution after consuming the last token and drafts
 * 0..i-1); t_i = argmax of row i (lowest index on ties, NaN never wins, an
 * all-NaN row gives 0).  n_accept[b] = the largest k <= N with
 * drafts[b, j] == t_j for all j < k; out_tokens[b] = drafts[b, 0..k-1], t_k,
 * then -1 up to 1+N entries.  drafts [B, N] int32, out_tokens [B, 1+N] int32,
 * out_n_accept [B] int32.  0 <= N, B >= 1, V >= 1. */
int mtp_verify_greedy(const void *logits, int ldtype, int B, int N, int V,
                      const int32_t *drafts, int32_t *out_tokens, int32_t *out_n_accept,
                      void *ws, size_t ws_bytes, mtp_stream_t stream);

/* Exact speculative sampling ([SP] item 4), B <= MTP_MAX_VERIFY_BATCH
 * sequences.  For row i < N of sequence b:
 * p_i = sample_dist(target row i), q_i = sample_dist(draft row i), both with
 * penalty set hist[b] u {drafts[b, 0..i-1]}; x = drafts[b, i] is accepted iff
 * u < p_i(x) / q_i(x) (u of counter (b, 4i + 1, ...)).  At the first
 * rejection the emitted token is drawn from norm(max(p_i - q_i, 0)) (from p_i
 * if that is empty) with u of (b, 4i + 2, ...) and the window ends; when all
 * N drafts are accepted the bonus token is drawn from p_N with u of
 * (b, 4N + 3, ...).  Draws walk the candidates in (probability desc, id asc)
 * order.  Uniforms: Philox-4x32-10, counter (b, 4i + purpose, offset lo,
 * offset hi), key (seed lo, seed hi), u = (word0 >> 8) * 2^-24.
 *   tgt_logits [B, 1+N, V], dft_logits [B, N, V] in ldtype; drafts [B, N];
 *   hist [B, H] int32 (newest last, entries < 0 ignored; NULL when H == 0);
 *   sp host pointer (temp > 0, top_k == 0); out_tokens [B, 1+N] (-1 padded);
 *   out_n_accept [B].  sample_dist's weights are exp(l - lmax) rounded once
 *   to fp32 (the exponential in fp64); every other step feeding a decision
 *   is IEEE fp32 in the order written above, sums sequential in (w desc,
 *   id asc) order.  A row whose min-p set exceeds 4096 candidates sets
 *   MTP_ERR_CAPACITY in the status word.  One launch (plus a memset of the
 *   workspace's counters); one pass over the logits. */
int mtp_verify_sample(const void *tgt_logits, const void *dft_logits, int ldtype,
                      int B, int N, int V, const int32_t *drafts,
                      const int32_t *hist, int H, const mtp_sample_params *sp,
                      uint64_t seed, uint64_t offset,
                      int32_t *out_tokens, int32_t *out_n_accept,
                      void *ws, size_t ws_bytes, mtp_stream_t stream);

/* Draws of a sampling drafter ([SP] item 4: the token drafted at window
 * position i is a draw from q_i = sample_dist(draft row i)).  For every
 * sequence b and i = 0..N-1 in order: q_i = sample_dist(dft_logits[b, i]) with
 * penalty set hist[b] u {out_drafts[b, 0..i-1]}, and out_drafts[b, i] = the
 * inverse-CDF pick of q_i with the uniform of counter (b, 4i + 0, offset lo,
 * offset hi), key (seed lo, seed hi) -- the same draw mtp_draft_block makes
 * at temp > 0, so mtp_verify_sample can then check these drafts exactly.
 *   dft_logits [B, N, V] in ldtype; hist [B, H] int32 (NULL when H == 0);
 *   sp host pointer (as for mtp_verify_sample); out_drafts [B, N] int32.
 * 1 <= N <= 16, B <= MTP_MAX_VERIFY_BATCH.  N launches (window position i
 * depends on the draws before it) plus one workspace memset. */
int mtp_sample_drafts(const void *dft_logits, int ldtype, int B, int N, int V,
                      const int32_t *hist, int H, const mtp_sample_params *sp,
                      uint64_t seed, uint64_t offset, int32_t *out_drafts,
                      void *ws, size_t ws_bytes, mtp_stream_t stream);

/* Greedy verify without a workspace.  The pages have no counterpart of this
 * call; it exists for callers that may not allocate device memory at all --
 * for example a serving loop that has already handed every byte of the GPU to
 * its weights and KV cache and forbids further allocations, or code that must
 * not call cudaMalloc because it can synchronize the device in the middle of a
 * decode step.  Same arguments, results and errors as mtp_verify_greedy, minus
 * `ws` / `ws_bytes`: the scratch is a 4 KiB array built into the library (held
 * on every GPU that loads it until the process exits), so B * (1 + N) may be
 * at most 480; larger sizes return MTP_ERR_UNSUPPORTED and launch nothing.
 * Allocates nothing.  The first call on a device looks up the array's device
 * address (with that device current); make that first call before any stream
 * capture.  All calls share the one array and every call clears it first, so
 * calls that may overlap on the GPU (different streams, or several host
 * threads) race and must be serialized by the caller.  The looked-up address
 * is kept for the life of the process: do not use this call on a device after
 * cudaDeviceReset() in the same process. */
int mtp_verify_greedy_noalloc(const void *logits, int ldtype, int B, int N, int V,
                              const int32_t *drafts, int32_t *out_tokens, int32_t *out_n_accept,
                              mtp_stream_t stream);

/* Device status of the most recent call that used `ws`: MTP_OK,
 * MTP_ERR_TIMEOUT or MTP_ERR_CAPACITY.  SYNCHRONIZES `stream` (a 4-byte
 * device-to-host copy).  Returns MTP_ERR_CUDA if the copy fails. */
int mtp_last_error(const void *ws, mtp_stream_t stream);

/* Static description of an error code. */
const char *mtp_strerror(int code);

/* Fault-detection check: launches the grid barrier of the draft kernel with
 * an arrival count that can never be reached and a wait limit of
 * `timeout_us` microseconds (1..1000000).  Every block gives up, the status
 * word becomes MTP_ERR_TIMEOUT and the kernel returns; the context stays
 * usable.  For tests of the timeout path; computes nothing. */
int mtp_debug_barrier_timeout(void *ws, size_t ws_bytes, int timeout_us, mtp_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MTP_H */
