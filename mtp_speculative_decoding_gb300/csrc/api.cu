// api.cu -- the C ABI declared in include/mtp.h: argument checks, workspace
// layout and launches.  No allocation, no synchronization (except
// mtp_last_error), no state kept between calls beyond a per-device cache of
// the SM count.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <math.h>
#include <string.h>

#include <mutex>

#include "common.cuh"
#include "draft.cuh"
#include "mtp.h"
#include "verify.cuh"

using namespace mtp;

namespace {

constexpr unsigned long long kBarrierLimitNs = 1000000000ull;  // 1 s per barrier wait

size_t al256(size_t x) { return (x + 255) & ~(size_t)255; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int num_sms() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    static int cache[64] = {0};
    if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 64) cache[dev] = n;
    return n;
}

// LM head on tensor cores: the dense head, bf16 weights and a batch of at
// least kTcMinBatch
bool tc_head_eligible(const mtp_config* c, int B) {
    return c->wdtype == MTP_DTYPE_BF16 && B >= kTcMinBatch && c->n_centroids == 0 && c->wquant == MTP_WQ_NONE;
}

// centroid-routed head: shared memory of its per-CTA sort (keys over n_c
// rounded up to a power of two, the rank sort's scratch, the selection)
size_t cent_smem(const mtp_config* c) {
    size_t P = 1;
    while (P < (size_t)c->n_centroids) P <<= 1;
    return (P + kRankSortMax) * sizeof(unsigned long long) + (size_t)c->centroid_top_k * sizeof(int);
}
int pad16(int B) { return (B + 15) & ~15; }

size_t draft_smem(const mtp_config* c, int B, int act_smem);
constexpr size_t kSmemLimit = 220 * 1024;

// Projections on tensor cores: eligible for the head path, activations
// staged in global memory, FFN width a multiple of the 128-row tile (the
// gate and up rows of one tile come from one matrix)
bool tc_proj_eligible(const mtp_config* c, int B) {
    return tc_head_eligible(c, B) && draft_smem(c, B, 1) > kSmemLimit && c->d_ff % kTcTileM == 0;
}

// split-K factors of the projection phases (PH_PRE .. PH_POST) for a grid of
// `grid` CTAs, and the floats of the largest split-partial set (nextn: the
// fused query / key / value projection in PH_Q)
struct TcPlan {
    int sk[6];
    size_t pb_floats;
};
TcPlan tc_plan(const mtp_config* c, int B, int grid, bool nextn) {
    TcPlan t;
    const size_t qd = (size_t)c->n_q_heads * c->head_dim;
    const size_t qr = (size_t)(nextn ? c->n_q_heads + 2 * c->n_kv_heads : c->n_q_heads) * c->head_dim;   // Q's rows
    const size_t R[6] = {(size_t)c->d_a, qr, (size_t)c->d_a, 2 * (size_t)c->d_ff, (size_t)c->d_a, (size_t)c->d_t};
    const size_t K[6] = {2 * (size_t)c->d_t, (size_t)c->d_a, qd, (size_t)c->d_a, (size_t)c->d_ff, (size_t)c->d_a};
    t.pb_floats = 0;
    for (int ph = 0; ph < 6; ++ph) {
        const int ntiles = (int)((R[ph] + kTcTileM - 1) / kTcTileM), nks = (int)((K[ph] + kTcTileK - 1) / kTcTileK);
        int S = grid / ntiles;
        if (S < 1 || ph == PH_POST) S = 1;   // the post-projection writes h directly
        if (S > nks) S = nks;
        const int kps = (nks + S - 1) / S;
        S = (nks + kps - 1) / kps;
        t.sk[ph] = S;
        if (ph != PH_POST && (size_t)S * B * R[ph] > t.pb_floats) t.pb_floats = (size_t)S * B * R[ph];
    }
    return t;
}
int draft_grid() {
    const int sms = num_sms();
    return sms < kMaxGrid ? sms : kMaxGrid;
}

struct DraftLayout {
    size_t att_cnt, SROW, amax, XB, XM, QR, OB, YB, MB, Y2, HN, HX, CL, PART, CONF, ROPE, ROPEQ, XH, XL, XA, XAL, PB, ZB, SBUF,
        ACT, end;
    int kmax;
};

// survivor capacity of a sampled row and kept-set capacity, for V tokens
int sample_rcap(long long V) { return (int)(V < kRowBufCap ? ((V + 7) & ~7LL) : kRowBufCap); }
int sample_ccap(long long V) { return (int)(V < kCandCap ? ((V + 7) & ~7LL) : kCandCap); }

int draft_kmax(const mtp_config* c) {
    int k = 2 * c->d_t;
    const int q = c->n_q_heads * c->head_dim;
    if (c->d_a > k) k = c->d_a;
    if (q > k) k = q;
    if (c->d_ff > k) k = c->d_ff;
    return k;
}

DraftLayout draft_layout(const mtp_config* c, int B, int N) {
    DraftLayout L;
    size_t off = sizeof(WsHeader);
    const size_t f = sizeof(float);
    const int grp = c->n_q_heads / c->n_kv_heads;
    L.kmax = draft_kmax(c);
    L.att_cnt = off; off = al256(off + (size_t)B * c->n_kv_heads * sizeof(unsigned int));
    L.SROW = off;    off = al256(off + 4 * (size_t)B * sizeof(unsigned int));   // zeroed with the header
    L.amax = off;    off = al256(off + (size_t)N * B * sizeof(unsigned long long));
    L.XB = off;      off = al256(off + (size_t)B * c->d_a * f);
    L.XM = off;      off = al256(off + (size_t)B * c->d_a * f);
    // query rows, and (NextN's fused projection) its key and value rows
    L.QR = off;      off = al256(off + (size_t)B * (c->n_q_heads + 2 * c->n_kv_heads) * c->head_dim * f);
    L.OB = off;      off = al256(off + (size_t)B * c->n_q_heads * c->head_dim * f);
    L.YB = off;      off = al256(off + (size_t)B * c->d_a * f);
    L.MB = off;      off = al256(off + (size_t)B * c->d_ff * f);
    L.Y2 = off;      off = al256(off + (size_t)B * c->d_a * f);
    L.HN = off;      off = al256(off + (size_t)B * c->d_t * f);
    L.HX = off;      off = al256(off + (size_t)B * c->d_t * f);   // NextN: the block output chain
    L.CL = off;      off = al256(off + (size_t)B * c->n_centroids * f);
    const size_t items = 2 * (size_t)kMaxGrid + (size_t)B * c->n_kv_heads;
    L.PART = off;    off = al256(off + items * attn_psz(grp, c->head_dim) * f);
    L.CONF = off;    off = al256(off + (size_t)kMaxGrid * B * 2 * f);
    L.ROPE = off;    off = al256(off + (size_t)MTP_MAX_VIEWS * (c->head_dim / 2) * sizeof(double));
    L.ROPEQ = off;   off = al256(off + (size_t)B * MTP_MAX_VIEWS * (c->head_dim / 2) * 2 * f);
    // tensor-core operands: K blocks of 64 columns x (kTcHeadM rows for the
    // head's h, Bp rows for the projections' inputs), bf16
    const size_t xb = tc_head_eligible(c, B) ? (size_t)((c->d_t + 63) / 64) * kTcHeadM * 128 : 0;
    L.XH = off;      off = al256(off + xb);
    L.XL = off;      off = al256(off + xb);
    const bool tcp = tc_proj_eligible(c, B);
    const size_t xa = tcp ? (size_t)((L.kmax + 63) / 64) * pad16(B) * 128 : 0;
    L.XA = off;      off = al256(off + xa);
    L.XAL = off;     off = al256(off + xa);
    size_t pbf = 0;   // the larger of the assistant's and the NextN drafter's split partials
    if (tcp) {
        const size_t a = tc_plan(c, B, draft_grid(), false).pb_floats, n = tc_plan(c, B, draft_grid(), true).pb_floats;
        pbf = a > n ? a : n;
    }
    L.PB = off;      off = al256(off + pbf * f);
    // sampled drafting: the step's logits and the sampler's per-row state
    L.ZB = off;      off = al256(off + (size_t)B * c->vocab * f);
    L.SBUF = off;    off = al256(off + (size_t)B * sample_rcap(c->vocab) * sizeof(int2));
    L.ACT = off;     off = al256(off + (size_t)B * L.kmax * f);
    L.end = off;
    return L;
}

// cuTensorMapEncodeTiled from the driver, resolved once
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// 2-D bf16 tensor map over a row-major [rows, cols] matrix: box of 64
// columns (128 bytes, 128-byte swizzle) by box_rows rows; out-of-range rows
// and columns read as zero
bool encode_bf16_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct GreedyLayout { size_t amax, end; };
GreedyLayout greedy_layout(int B, int N) {
    GreedyLayout L;
    L.amax = sizeof(WsHeader);
    L.end = al256(L.amax + (size_t)B * (N + 1) * sizeof(unsigned long long));
    return L;
}

// Sampler workspace: the per-row state (4 x rows words) and the
// per-sequence counters, zeroed before a launch, then the survivor buffers
// and (verification) the kept sets.
struct SampleLayout { size_t row, seq, ctr, zero_end, buf, nkeep, wkeep, id, w, end; };
SampleLayout sample_layout(long long rows, int B, long long V, bool verify) {
    SampleLayout L;
    size_t off = sizeof(WsHeader);
    L.row = off;   off += 4 * (size_t)rows * sizeof(unsigned int);
    L.seq = off;   off += (size_t)B * sizeof(unsigned int);
    L.ctr = off;   off += sizeof(unsigned int);
    L.zero_end = off;
    off = al256(off);
    L.buf = off;   off = al256(off + (size_t)rows * sample_rcap(V) * sizeof(int2));
    const size_t kr = verify ? (size_t)rows : 0, cc = verify ? (size_t)sample_ccap(V) : 0;
    L.nkeep = off; off = al256(off + kr * sizeof(int32_t));
    L.wkeep = off; off = al256(off + kr * sizeof(float));
    L.id = off;    off = al256(off + kr * cc * sizeof(int32_t));
    L.w = off;     off = al256(off + kr * cc * sizeof(float));
    L.end = off;
    return L;
}
long long verify_rows(int B, int N) { return (long long)B * (N + 1) + (long long)B * N; }

// residual scratch plus staged activations of the GEMV phases
size_t draft_smem_act(const mtp_config* c, int B, int act_smem) {
    const size_t kmax = draft_kmax(c), gmax = (size_t)(c->d_t > c->d_a ? c->d_t : c->d_a);
    return (((size_t)c->d_a + 3) & ~(size_t)3) * sizeof(float) +
           (act_smem ? (size_t)B * kmax : kmax) * sizeof(float) + 2 * gmax * sizeof(float);   // + the gain stage
}

size_t draft_smem(const mtp_config* c, int B, int act_smem) {
    const size_t wb = c->wdtype == MTP_DTYPE_BF16 ? 2 : 4;
    const size_t hd = c->head_dim, grp = c->n_q_heads / c->n_kv_heads;
    const int nst = tc_head_eligible(c, B) ? kAttnStagesTc : kAttnStages;   // the kernel variant's ring depth
    const size_t attn = attn_smem((int)hd, (int)wb, (int)grp, nst);
    const size_t act = draft_smem_act(c, B, act_smem);
    return attn > act ? attn : act;
}

// floor(2^32 / n) for n >= 2 (2^32 - 1 for n = 1): the device's
// multiply-high modulo (ring_mod) is then exact after one correction
unsigned int mod_magic(unsigned int n) {
    return n <= 1 ? 0xFFFFFFFFu : (unsigned int)(0x100000000ull / (unsigned long long)n);
}

int check_config(const mtp_config* c) {
    if (!c) return MTP_ERR_ARG;
    if (c->d_t <= 0 || c->d_a <= 0 || c->n_blocks <= 0 || c->n_q_heads <= 0 || c->head_dim <= 0 ||
        c->n_kv_heads <= 0 || c->d_ff <= 0 || c->vocab <= 0)
        return MTP_ERR_ARG;
    if (c->n_blocks > MTP_MAX_BLOCKS) return MTP_ERR_UNSUPPORTED;
    if (c->n_q_heads % c->n_kv_heads != 0) return MTP_ERR_ARG;
    if (c->n_q_heads / c->n_kv_heads > 16) return MTP_ERR_UNSUPPORTED;
    if (c->wdtype != MTP_DTYPE_F32 && c->wdtype != MTP_DTYPE_BF16) return MTP_ERR_UNSUPPORTED;
    const int hd = c->head_dim;
    if (hd != 32 && hd != 64 && hd != 128 && hd != 256 && hd != 512) return MTP_ERR_UNSUPPORTED;
    const int m = 8;  // row lengths in elements: 16-byte rows for either dtype
    if (c->d_t % m || c->d_a % m || c->d_ff % m || (c->n_q_heads * hd) % m) return MTP_ERR_UNSUPPORTED;
    if (!(c->rms_eps >= 0.f) || !(c->attn_scale >= 0.f) || !(c->emb_scale >= 0.f) || !(c->logit_softcap >= 0.f))
        return MTP_ERR_ARG;
    if (c->n_centroids < 0 || c->centroid_top_k < 0) return MTP_ERR_ARG;
    if (c->wquant != MTP_WQ_NONE && c->wquant != MTP_WQ_Q8_0 && c->wquant != MTP_WQ_Q4_0) return MTP_ERR_UNSUPPORTED;
    if (c->wquant != MTP_WQ_NONE) {
        if (c->wdtype != MTP_DTYPE_BF16 || (hd != 64 && hd != 128 && hd != 256)) return MTP_ERR_UNSUPPORTED;
        if (c->d_t % 32 || c->d_a % 32 || c->d_ff % 32 || (c->n_q_heads * hd) % 32) return MTP_ERR_UNSUPPORTED;
    }
    if (c->n_centroids > 0) {
        if (c->n_centroids > MTP_MAX_CENTROIDS) return MTP_ERR_UNSUPPORTED;
        if (c->centroid_top_k < 1 || c->centroid_top_k > c->n_centroids || c->vocab % c->n_centroids) return MTP_ERR_ARG;
    }
    return MTP_OK;
}

int check_workspace(const void* ws, size_t ws_bytes, size_t need) {
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255) != 0) return MTP_ERR_WORKSPACE;
    if (ws_bytes < need) return MTP_ERR_WORKSPACE;
    return MTP_OK;
}

int check_sample_params(const mtp_sample_params* sp) {
    if (!sp) return MTP_ERR_ARG;
    if (!(sp->temp > 0.f) || !(sp->top_p > 0.f) || !(sp->min_p >= 0.f) || sp->min_p > 1.f ||
        !(sp->rep_penalty > 0.f) || sp->presence_penalty != sp->presence_penalty)
        return MTP_ERR_ARG;
    if (sp->top_k != 0) return MTP_ERR_UNSUPPORTED;
    return MTP_OK;
}

// the sampler's job for either entry point (mode, rows and outputs set by the caller)
SampleJob sample_job(const void* base0, const void* base1, int ldtype, int B, int N, int V, const int32_t* drafts,
                     const int32_t* hist, int H, const mtp_sample_params* sp, uint64_t seed, uint64_t offset,
                     char* ws, const SampleLayout& L, long long rows, int sms) {
    SampleJob j;
    memset(&j, 0, sizeof j);
    j.base0 = base0;
    j.base1 = base1;
    j.f32 = ldtype == MTP_DTYPE_F32;
    j.B = B;
    j.N = N;
    j.V = V;
    j.drafts = drafts;
    j.drafts_ld = N;
    j.hist = hist;
    j.H = H;
    j.hist_ld = H;
    j.temp = sp->temp; j.top_p = sp->top_p; j.min_p = sp->min_p; j.rep = sp->rep_penalty;
    j.pres = sp->presence_penalty;
    j.seed = seed;
    j.offset = offset;
    j.hdr = reinterpret_cast<WsHeader*>(ws);
    unsigned int* row = reinterpret_cast<unsigned int*>(ws + L.row);
    j.row_max = row;
    j.row_cnt = row + rows;
    j.row_ovf = row + 2 * rows;
    j.row_done = row + 3 * rows;
    j.seq_done = reinterpret_cast<unsigned int*>(ws + L.seq);
    j.next_piece = reinterpret_cast<unsigned int*>(ws + L.ctr);
    j.row_buf = reinterpret_cast<int2*>(ws + L.buf);
    j.rcap = sample_rcap(V);
    j.keep_id = reinterpret_cast<int32_t*>(ws + L.id);
    j.keep_w = reinterpret_cast<float*>(ws + L.w);
    j.ccap = sample_ccap(V);
    j.n_keep = reinterpret_cast<int32_t*>(ws + L.nkeep);
    j.w_keep = reinterpret_cast<float*>(ws + L.wkeep);
    const int per_sm = sample_blocks_per_sm();
    sample_piece_plan(V, rows, (per_sm > 0 ? per_sm : 1) * sms, &j.ppr, &j.piece_len);
    return j;
}

int check_logits(const void* a, const void* b, int ldtype) {
    if (ldtype != MTP_DTYPE_F32 && ldtype != MTP_DTYPE_BF16) return MTP_ERR_UNSUPPORTED;
    const uintptr_t am = ldtype == MTP_DTYPE_BF16 ? 1 : 3;
    if ((reinterpret_cast<uintptr_t>(a) & am) || (b && (reinterpret_cast<uintptr_t>(b) & am))) return MTP_ERR_ARG;
    return MTP_OK;
}

}  // namespace

extern "C" {

int mtp_quantize_q8_0(const float* w, int64_t rows, int64_t cols, int8_t* codes, uint16_t* scales) {
    if (!w || !codes || !scales || rows < 0 || cols < 0 || cols % 32) return MTP_ERR_ARG;
    const int64_t nb = cols / 32;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t j = 0; j < nb; ++j) {
            const float* x = w + r * cols + j * 32;
            float amax = 0.f;
            for (int i = 0; i < 32; ++i) {
                const float a = fabsf(x[i]);
                if (a > amax) amax = a;
            }
            const float d = amax / 127.f;
            const float inv = d != 0.f ? 1.f / d : 0.f;
            int8_t* q = codes + r * cols + j * 32;
            for (int i = 0; i < 32; ++i) q[i] = (int8_t)roundf(x[i] * inv);
            scales[r * nb + j] = __half_as_ushort(__float2half_rn(d));
        }
    }
    return MTP_OK;
}

int mtp_quantize_q4_0(const float* w, int64_t rows, int64_t cols, uint8_t* codes, uint16_t* scales) {
    if (!w || !codes || !scales || rows < 0 || cols < 0 || cols % 32) return MTP_ERR_ARG;
    const int64_t nb = cols / 32;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t j = 0; j < nb; ++j) {
            const float* x = w + r * cols + j * 32;
            float amax = 0.f, m = 0.f;   // the first weight of largest magnitude, with its sign
            for (int i = 0; i < 32; ++i) {
                const float a = fabsf(x[i]);
                if (a > amax) {
                    amax = a;
                    m = x[i];
                }
            }
            const float d = m / -8.f;
            const float inv = d != 0.f ? 1.f / d : 0.f;
            uint8_t* q = codes + r * (cols / 2) + j * 16;
            for (int i = 0; i < 16; ++i) {
                const int lo = (int)(x[i] * inv + 8.5f), hi = (int)(x[i + 16] * inv + 8.5f);   // truncations
                q[i] = (uint8_t)((lo < 15 ? lo : 15) | ((hi < 15 ? hi : 15) << 4));
            }
            scales[r * nb + j] = __half_as_ushort(__float2half_rn(d));
        }
    }
    return MTP_OK;
}

size_t mtp_workspace_size(const mtp_config* cfg, int B, int N, int V) {
    if (B <= 0 || B > MTP_MAX_VERIFY_BATCH || N < 0 || N > 16 || V <= 0) return 0;
    if (cfg && B > MTP_MAX_BATCH) return 0;
    size_t need = al256(greedy_layout(B, N).end);
    const size_t s = sample_layout(verify_rows(B, N), B, V, true).end;
    if (s > need) need = s;
    if (cfg) {
        if (check_config(cfg) != MTP_OK || N < 1) return 0;
        const size_t d = draft_layout(cfg, B, N).end;
        if (d > need) need = d;
    }
    return need;
}

}  // extern "C"

namespace {

// NextN's extra inputs (null for the assistant)
struct NextnIn {
    const int32_t* n_cu;
    const int32_t* cu_tok;
    const float* cu_h;
    int M;
};

// mtp_draft_block, and mtp_nextn_draft when nx != null: the checks, the
// parameter block and the launch of the persistent draft kernel
int draft_impl(const mtp_config* cfg, const mtp_weights* w, const mtp_kv_view* views, int n_views,
               const int32_t* kv_len, int B, int N, const int32_t* last_tok, const float* h_prev,
               const mtp_sample_params* sp, uint64_t seed, uint64_t offset, const int32_t* hist, int H,
               int32_t* out_drafts, float* out_h_last, float* out_logits, float* out_conf, void* ws,
               size_t ws_bytes, mtp_stream_t stream, const NextnIn* nx) {
    int rc = check_config(cfg);
    if (rc != MTP_OK) return rc;
    if (nx) {
        if (cfg->d_a != cfg->d_t) return MTP_ERR_ARG;
        if (cfg->n_blocks != 1 || cfg->n_centroids != 0) return MTP_ERR_UNSUPPORTED;
        if (nx->M < 0 || nx->M > MTP_MAX_CATCHUP) return MTP_ERR_ARG;
        if (nx->M > 0 && (!nx->cu_tok || !nx->cu_h)) return MTP_ERR_ARG;
        if ((reinterpret_cast<uintptr_t>(nx->cu_h) & 3) || (reinterpret_cast<uintptr_t>(nx->cu_tok) & 3) ||
            (reinterpret_cast<uintptr_t>(nx->n_cu) & 3))
            return MTP_ERR_ARG;
        if (n_views != 1 || !views || views[0].window != 0 || views[0].sink != 0) return MTP_ERR_ARG;
        if (sp) return MTP_ERR_ARG;
    }
    if (!w || !views || n_views < 1 || n_views > MTP_MAX_VIEWS) return MTP_ERR_ARG;
    if (B < 1 || B > MTP_MAX_BATCH || N < 1 || N > 16) return MTP_ERR_ARG;
    if (!kv_len || !last_tok || !h_prev || !out_drafts) return MTP_ERR_ARG;
    if (H < 0 || (H > 0 && !hist)) return MTP_ERR_ARG;
    const bool sampling = sp && sp->temp > 0.f;
    if (sampling) {
        const int rs = check_sample_params(sp);
        if (rs != MTP_OK) return rs;
        if (H < 0 || (H > 0 && !hist)) return MTP_ERR_ARG;
    }
    const bool bf = cfg->wdtype == MTP_DTYPE_BF16;
    const int esz = bf ? 2 : 4;
    // weights
    const void* mats[] = {w->tok_embd, w->w_pre, nx ? w->tok_embd : w->w_post};   // NextN has no post-projection
    for (const void* m : mats) if (!m || !aligned16(m)) return MTP_ERR_ARG;
    if (cfg->wquant != MTP_WQ_NONE) {
        const uint16_t* sc[] = {w->w_pre_scale, nx ? w->w_pre_scale : w->w_post_scale};   // NextN: no post-projection
        for (const uint16_t* x : sc) if (!x || (reinterpret_cast<uintptr_t>(x) & 1)) return MTP_ERR_ARG;
        for (int l = 0; l < cfg->n_blocks; ++l) {
            const mtp_block_weights& b = w->blk[l];
            const uint16_t* bs[] = {b.w_q_scale, b.w_o_scale, b.w_gate_scale, b.w_up_scale, b.w_down_scale};
            for (const uint16_t* x : bs) if (!x || (reinterpret_cast<uintptr_t>(x) & 1)) return MTP_ERR_ARG;
        }
    }
    const bool cent = cfg->n_centroids > 0;
    if (cent && (!w->centroids || !aligned16(w->centroids) || !w->token_ordering ||
                 (reinterpret_cast<uintptr_t>(w->token_ordering) & 3)))
        return MTP_ERR_ARG;
    if (!w->norm_e || !w->norm_h || !w->final_norm) return MTP_ERR_ARG;
    for (int l = 0; l < cfg->n_blocks; ++l) {
        const mtp_block_weights& b = w->blk[l];
        const void* bm[] = {b.w_q, b.w_o, b.w_gate, b.w_up, b.w_down};
        for (const void* m : bm) if (!m || !aligned16(m)) return MTP_ERR_ARG;
        if (!b.attn_norm || !b.q_norm || !b.pre_ffn_norm) return MTP_ERR_ARG;
        if (nx ? !b.k_norm : (!b.post_attn_norm || !b.post_ffn_norm)) return MTP_ERR_ARG;
        if (!nx && (b.kv_view < 0 || b.kv_view >= n_views)) return MTP_ERR_ARG;
    }
    for (int v = 0; v < n_views; ++v) {
        const mtp_kv_view& kv = views[v];
        if (!kv.k || !kv.v || !aligned16(kv.k) || !aligned16(kv.v)) return MTP_ERR_ARG;
        if (kv.cap < 1 || kv.window < 0 || kv.window > kv.cap || !(kv.rope_theta > 0.f)) return MTP_ERR_ARG;
        if (kv.sink < 0 || (kv.window == 0 && kv.sink != 0) || (long long)kv.window + kv.sink > kv.cap)
            return MTP_ERR_ARG;
        if (kv.stride_t < cfg->head_dim || kv.stride_b < 0 || kv.stride_h < 0) return MTP_ERR_ARG;
        if ((kv.stride_t * esz) % 16 || (kv.stride_h * esz) % 16 || (kv.stride_b * esz) % 16) return MTP_ERR_ARG;
    }
    const DraftLayout L = draft_layout(cfg, B, N);
    rc = check_workspace(ws, ws_bytes, L.end);
    if (rc != MTP_OK) return rc;
    const int sms = num_sms();
    if (sms <= 0) return MTP_ERR_CUDA;

    size_t smem = draft_smem(cfg, B, 1);
    int act_smem = 1;
    if (smem > kSmemLimit) {
        act_smem = 0;
        smem = draft_smem(cfg, B, 0);
        if (smem > kSmemLimit) return MTP_ERR_UNSUPPORTED;
    }
    const int grid = draft_grid();
    // one sequence: LM head rows through bulk-copy slots at offset 0
    int head_slotb = 0;
    if (!cent && B == 1 && (size_t)cfg->d_t * esz / 16 <= (size_t)kHeadMaxChunks) {
        const size_t slotb = ((size_t)cfg->d_t * esz + 127) & ~(size_t)127;
        const size_t ring = (size_t)kHeadGroups * kHeadSlots * slotb;
        if (ring <= kSmemLimit) {
            head_slotb = (int)slotb;
            if (ring > smem) smem = ring;
        }
    }
    // batch: LM head on tensor cores, operand ring at offset 0 (1024-aligned)
    const bool tc = tc_head_eligible(cfg, B);
    int tc_stages = 0, tc_cols = 0, th_stages = 0;
    if (tc) {
        const size_t sbytes = (size_t)kTcTileM * 128 + 2 * (size_t)pad16(B) * 128;
        tc_stages = (int)(kTcSmemBudget / sbytes);
        if (tc_stages > kTcMaxStages) tc_stages = kTcMaxStages;
        if (tc_stages < 2) return MTP_ERR_UNSUPPORTED;
        size_t need = (size_t)tc_stages * sbytes + 1024 + kTcStageBytes;   // ring + epilogue staging
        if (need > smem) smem = need;
        // the head's ring: a table box and h's high (and, sampling, low) block per stage
        const size_t hbytes = (size_t)kTcHeadN * 128 + (sampling ? 2 : 1) * (size_t)kTcHeadM * 128;
        th_stages = (int)(kTcHeadSmemBudget / hbytes);
        if (th_stages > kTcMaxStages) th_stages = kTcMaxStages;
        need = (size_t)th_stages * hbytes + 1024;
        if (need > smem) smem = need;
        tc_cols = kTcHeadCols;   // the head's two accumulators; the projections use the first 2 Bp columns
    }
    if (cent && cent_smem(cfg) > smem) smem = cent_smem(cfg);   // at most 100 KB (n_c <= MTP_MAX_CENTROIDS)
    const bool q8 = cfg->wquant == MTP_WQ_Q8_0, q4 = cfg->wquant == MTP_WQ_Q4_0;
    const int per_sm = !bf ? draft_blocks_per_sm_f32(cfg->head_dim, smem)
                       : tc ? draft_blocks_per_sm_bf16_tc(cfg->head_dim, smem)
                       : q8 ? draft_blocks_per_sm_q8(cfg->head_dim, smem)
                       : q4 ? draft_blocks_per_sm_q4(cfg->head_dim, smem)
                            : draft_blocks_per_sm_bf16_cc(cfg->head_dim, smem);
    if (per_sm < 1) return MTP_ERR_UNSUPPORTED;

    char* base = static_cast<char*>(ws);
    DraftParams p;
    memset(&p, 0, sizeof p);
    p.d_t = cfg->d_t; p.d_a = cfg->d_a; p.L = cfg->n_blocks; p.Hq = cfg->n_q_heads; p.hd = cfg->head_dim;
    p.Hkv = cfg->n_kv_heads; p.F = cfg->d_ff; p.V = cfg->vocab; p.B = B; p.N = N;
    p.eps = cfg->rms_eps; p.softcap = cfg->logit_softcap;
    // 0 selects the defaults the header documents: 1/sqrt(head_dim), sqrt(d_t)
    p.attn_scale = cfg->attn_scale > 0.f ? cfg->attn_scale : (float)(1.0 / sqrt((double)cfg->head_dim));
    p.emb_scale = cfg->emb_scale > 0.f ? cfg->emb_scale : nx ? 1.f : (float)sqrt((double)cfg->d_t);
    p.tok_embd = w->tok_embd;
    p.norm_e = static_cast<const float*>(w->norm_e);
    p.norm_h = static_cast<const float*>(w->norm_h);
    p.w_pre = w->w_pre;
    p.final_norm = static_cast<const float*>(w->final_norm);
    p.w_post = w->w_post;
    if (cfg->wquant != MTP_WQ_NONE) {
        p.s_pre = w->w_pre_scale;
        p.s_post = nx ? nullptr : w->w_post_scale;
    }
    for (int l = 0; l < cfg->n_blocks; ++l) {
        const mtp_block_weights& b = w->blk[l];
        BlkW& d = p.blk[l];
        d.w_q = b.w_q; d.w_o = b.w_o; d.w_gate = b.w_gate; d.w_up = b.w_up; d.w_down = b.w_down;
        if (q8 || q4) {
            d.s_q = b.w_q_scale; d.s_o = b.w_o_scale; d.s_gate = b.w_gate_scale; d.s_up = b.w_up_scale;
            d.s_down = b.w_down_scale;
        }
        d.attn_norm = static_cast<const float*>(b.attn_norm);
        d.q_norm = static_cast<const float*>(b.q_norm);
        d.post_attn_norm = static_cast<const float*>(b.post_attn_norm);
        d.pre_ffn_norm = static_cast<const float*>(b.pre_ffn_norm);
        d.post_ffn_norm = static_cast<const float*>(b.post_ffn_norm);
        d.k_norm = nx ? static_cast<const float*>(b.k_norm) : nullptr;
        d.view = nx ? 0 : b.kv_view;
    }
    for (int v = 0; v < n_views; ++v) {
        KView& d = p.views[v];
        d.k = views[v].k; d.v = views[v].v;
        d.sb = views[v].stride_b; d.sh = views[v].stride_h; d.st = views[v].stride_t;
        d.cap = views[v].cap; d.window = views[v].window; d.theta = views[v].rope_theta; d.sink = views[v].sink;
        d.cap_magic = mod_magic((unsigned int)d.cap);
        d.ring_magic = mod_magic((unsigned int)(d.cap - (d.window > 0 ? d.sink : 0)));
    }
    p.kv_len = kv_len; p.last_tok = last_tok; p.h_prev = h_prev;
    p.QS = (nx ? cfg->n_q_heads + 2 * cfg->n_kv_heads : cfg->n_q_heads) * cfg->head_dim;
    if (nx) {
        p.nextn = 1;
        p.M = nx->M;
        p.n_cu = nx->M > 0 ? nx->n_cu : nullptr;
        p.cu_tok = nx->cu_tok;
        p.cu_h = nx->cu_h;
    }
    p.out_drafts = out_drafts; p.out_h_last = out_h_last; p.out_logits = out_logits; p.out_conf = out_conf;
    p.hdr = reinterpret_cast<WsHeader*>(base);
    p.att_cnt = reinterpret_cast<unsigned int*>(base + L.att_cnt);
    p.amax = reinterpret_cast<unsigned long long*>(base + L.amax);
    p.XB = reinterpret_cast<float*>(base + L.XB);
    p.XM = reinterpret_cast<float*>(base + L.XM);
    p.QR = reinterpret_cast<float*>(base + L.QR);
    p.OB = reinterpret_cast<float*>(base + L.OB);
    p.YB = reinterpret_cast<float*>(base + L.YB);
    p.MB = reinterpret_cast<float*>(base + L.MB);
    p.Y2 = reinterpret_cast<float*>(base + L.Y2);
    p.HN = reinterpret_cast<float*>(base + L.HN);
    p.HX = reinterpret_cast<float*>(base + L.HX);
    p.PART = reinterpret_cast<float*>(base + L.PART);
    p.CONF = reinterpret_cast<float2*>(base + L.CONF);
    p.ROPE = reinterpret_cast<double*>(base + L.ROPE);
    p.ROPEQ = reinterpret_cast<float2*>(base + L.ROPEQ);
    p.ACT = reinterpret_cast<float*>(base + L.ACT);
    if (cent) {
        p.n_cent = cfg->n_centroids;
        p.cent_k = cfg->centroid_top_k;
        p.cent = w->centroids;
        p.cord = w->token_ordering;
        p.CL = reinterpret_cast<float*>(base + L.CL);
    }
    p.act_smem = act_smem;
    p.head_slotb = head_slotb;
    if (tc) {
        p.tc_head = 1;
        p.Bp = pad16(B);
        p.tc_stages = tc_stages;
        p.th_stages = th_stages;
        p.tc_cols = tc_cols;
        p.XH = reinterpret_cast<uint16_t*>(base + L.XH);
        p.XL = reinterpret_cast<uint16_t*>(base + L.XL);
        if (!encode_bf16_map(&p.tm_embd, w->tok_embd, (uint64_t)cfg->d_t, (uint64_t)cfg->vocab, kTcHeadN))
            return MTP_ERR_CUDA;
        if (tc_proj_eligible(cfg, B) && !act_smem) {
            // projections: weights [R, K] row-major, inputs staged as [Bp, kmax]
            const TcPlan plan = tc_plan(cfg, B, grid, nx != nullptr);
            p.tc_proj = 1;
            p.att_fold = 1;   // the O prologue merges split attention segments: one row per CTA, no counter waits
            for (int i = 0; i < 6; ++i) p.sk[i] = plan.sk[i];
            p.XA = reinterpret_cast<uint16_t*>(base + L.XA);
            p.XAL = reinterpret_cast<uint16_t*>(base + L.XAL);
            p.PB = reinterpret_cast<float*>(base + L.PB);
            const uint64_t da = cfg->d_a, dt = cfg->d_t, F = cfg->d_ff, qd = (uint64_t)cfg->n_q_heads * cfg->head_dim;
            const uint64_t qr = (uint64_t)p.QS;   // rows of w_q: NextN's fused projection has the key and value rows too
            bool okm = encode_bf16_map(&p.tm_w[0], w->w_pre, 2 * dt, da, kTcTileM) &&
                       (nx || encode_bf16_map(&p.tm_w[1], w->w_post, da, dt, kTcTileM));   // NextN: no post-projection
            for (int l = 0; l < cfg->n_blocks && okm; ++l) {
                const mtp_block_weights& bw = w->blk[l];
                CUtensorMap* m = &p.tm_w[2 + 5 * l];
                okm = encode_bf16_map(m + 0, bw.w_q, da, qr, kTcTileM) && encode_bf16_map(m + 1, bw.w_o, qd, da, kTcTileM) &&
                      encode_bf16_map(m + 2, bw.w_gate, da, F, kTcTileM) &&
                      encode_bf16_map(m + 3, bw.w_up, da, F, kTcTileM) &&
                      encode_bf16_map(m + 4, bw.w_down, F, da, kTcTileM);
            }
            if (!okm) return MTP_ERR_CUDA;
        }
    }
    p.kmax = L.kmax;
    p.timeout_ns = kBarrierLimitNs;
    if (sampling) {
        p.sampling = 1;
        p.s_temp = sp->temp; p.s_top_p = sp->top_p; p.s_min_p = sp->min_p;
        p.s_rep = sp->rep_penalty; p.s_pres = sp->presence_penalty;
        p.seed = seed; p.offset = offset; p.hist = hist; p.H = H;
        p.ZB = reinterpret_cast<float*>(base + L.ZB);
        p.S_row = reinterpret_cast<unsigned int*>(base + L.SROW);
        p.S_buf = reinterpret_cast<int2*>(base + L.SBUF);
        p.S_rcap = sample_rcap(cfg->vocab);
        sample_piece_plan(cfg->vocab, B, grid, &p.S_ppr, &p.S_plen);
        if (smem < kSampleSmem) smem = kSampleSmem;
    }

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(ws, 0, L.amax, s) != cudaSuccess) return MTP_ERR_CUDA;
    cudaError_t e = !bf ? launch_draft_f32(p, grid, smem, s)
                    : p.tc_head ? launch_draft_bf16_tc(p, grid, smem, s)
                    : q8 ? launch_draft_q8(p, grid, smem, s)
                    : q4 ? launch_draft_q4(p, grid, smem, s)
                                : launch_draft_bf16_cc(p, grid, smem, s);
    return e == cudaSuccess ? MTP_OK : MTP_ERR_CUDA;
}

}  // namespace

extern "C" {

int mtp_draft_block(const mtp_config* cfg, const mtp_weights* w, const mtp_kv_view* views, int n_views,
                    const int32_t* kv_len, int B, int N, const int32_t* last_tok, const float* h_prev,
                    const mtp_sample_params* sp, uint64_t seed, uint64_t offset, const int32_t* hist, int H,
                    int32_t* out_drafts, float* out_h_last, float* out_logits, float* out_conf, void* ws,
                    size_t ws_bytes, mtp_stream_t stream) {
    return draft_impl(cfg, w, views, n_views, kv_len, B, N, last_tok, h_prev, sp, seed, offset, hist, H, out_drafts,
                      out_h_last, out_logits, out_conf, ws, ws_bytes, stream, nullptr);
}

int mtp_nextn_draft(const mtp_config* cfg, const mtp_weights* w, const mtp_kv_view* dkv, const int32_t* kv_len, int B,
                    int N, const int32_t* n_cu, const int32_t* cu_tok, const float* cu_h, int M,
                    const int32_t* last_tok, const float* h_prev, int32_t* out_drafts, float* out_h_last,
                    float* out_logits, float* out_conf, void* ws, size_t ws_bytes, mtp_stream_t stream) {
    if (!dkv) return MTP_ERR_ARG;
    const NextnIn nx{n_cu, cu_tok, cu_h, M};
    return draft_impl(cfg, w, dkv, 1, kv_len, B, N, last_tok, h_prev, nullptr, 0, 0, nullptr, 0, out_drafts,
                      out_h_last, out_logits, out_conf, ws, ws_bytes, stream, &nx);
}

int mtp_verify_greedy(const void* logits, int ldtype, int B, int N, int V, const int32_t* drafts, int32_t* out_tokens,
                      int32_t* out_n_accept, void* ws, size_t ws_bytes, mtp_stream_t stream) {
    if (!logits || !out_tokens || !out_n_accept) return MTP_ERR_ARG;
    if (B < 1 || B > MTP_MAX_VERIFY_BATCH || N < 0 || N > 16 || V < 1) return MTP_ERR_ARG;
    if (N > 0 && !drafts) return MTP_ERR_ARG;
    const int lc = check_logits(logits, nullptr, ldtype);
    if (lc != MTP_OK) return lc;
    const GreedyLayout L = greedy_layout(B, N);
    int rc = check_workspace(ws, ws_bytes, L.end);
    if (rc != MTP_OK) return rc;
    const int sms = num_sms();
    if (sms <= 0) return MTP_ERR_CUDA;
    char* base = static_cast<char*>(ws);
    VerifyGreedyArgs a;
    a.logits = logits; a.B = B; a.N = N; a.V = V; a.drafts = drafts;
    a.out_tokens = out_tokens; a.out_n_accept = out_n_accept;
    a.hdr = reinterpret_cast<WsHeader*>(base);
    a.amax = reinterpret_cast<unsigned long long*>(base + L.amax);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(ws, 0, L.end, s) != cudaSuccess) return MTP_ERR_CUDA;
    return launch_verify_greedy(a, ldtype, sms, s) == cudaSuccess ? MTP_OK : MTP_ERR_CUDA;
}

int mtp_verify_sample(const void* tgt_logits, const void* dft_logits, int ldtype, int B, int N, int V,
                      const int32_t* drafts, const int32_t* hist, int H, const mtp_sample_params* sp, uint64_t seed,
                      uint64_t offset, int32_t* out_tokens, int32_t* out_n_accept, void* ws, size_t ws_bytes,
                      mtp_stream_t stream) {
    if (!tgt_logits || !out_tokens || !out_n_accept) return MTP_ERR_ARG;
    if (B < 1 || B > MTP_MAX_VERIFY_BATCH || N < 0 || N > 16 || V < 1) return MTP_ERR_ARG;
    if (N > 0 && (!drafts || !dft_logits)) return MTP_ERR_ARG;
    if (H < 0 || (H > 0 && !hist)) return MTP_ERR_ARG;
    int rc = check_logits(tgt_logits, dft_logits, ldtype);
    if (rc != MTP_OK) return rc;
    rc = check_sample_params(sp);
    if (rc != MTP_OK) return rc;
    const long long rows = verify_rows(B, N);
    const SampleLayout L = sample_layout(rows, B, V, true);
    rc = check_workspace(ws, ws_bytes, L.end);
    if (rc != MTP_OK) return rc;
    const int sms = num_sms();
    if (sms <= 0) return MTP_ERR_CUDA;
    char* base = static_cast<char*>(ws);
    SampleJob j = sample_job(tgt_logits, dft_logits, ldtype, B, N, V, drafts, hist, H, sp, seed, offset, base, L,
                             rows, sms);
    j.mode = 0;
    j.out_tokens = out_tokens;
    j.out_n_accept = out_n_accept;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(ws, 0, L.zero_end, s) != cudaSuccess) return MTP_ERR_CUDA;
    return launch_sample(j, sms, s) == cudaSuccess ? MTP_OK : MTP_ERR_CUDA;
}

int mtp_sample_drafts(const void* dft_logits, int ldtype, int B, int N, int V, const int32_t* hist, int H,
                      const mtp_sample_params* sp, uint64_t seed, uint64_t offset, int32_t* out_drafts, void* ws,
                      size_t ws_bytes, mtp_stream_t stream) {
    if (!dft_logits || !out_drafts) return MTP_ERR_ARG;
    if (B < 1 || B > MTP_MAX_VERIFY_BATCH || N < 1 || N > 16 || V < 1) return MTP_ERR_ARG;
    if (H < 0 || (H > 0 && !hist)) return MTP_ERR_ARG;
    int rc = check_logits(dft_logits, nullptr, ldtype);
    if (rc != MTP_OK) return rc;
    rc = check_sample_params(sp);
    if (rc != MTP_OK) return rc;
    const SampleLayout L = sample_layout(B, B, V, false);
    rc = check_workspace(ws, ws_bytes, L.end);
    if (rc != MTP_OK) return rc;
    const int sms = num_sms();
    if (sms <= 0) return MTP_ERR_CUDA;
    char* base = static_cast<char*>(ws);
    SampleJob j = sample_job(dft_logits, nullptr, ldtype, B, N, V, out_drafts, hist, H, sp, seed, offset, base, L,
                             B, sms);
    j.mode = 1;
    j.draw_ld = (long long)N * V;
    j.out_draw = out_drafts;
    j.out_draw_ld = N;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // the row state is zeroed once; every row's finishing CTA re-zeroes it
    if (cudaMemsetAsync(ws, 0, L.zero_end, s) != cudaSuccess) return MTP_ERR_CUDA;
    const size_t esz = ldtype == MTP_DTYPE_BF16 ? 2 : 4;
    for (int i = 0; i < N; ++i) {   // draw i's penalty set holds draws 0..i-1: one launch per window position
        if (i > 0 && cudaMemsetAsync(j.next_piece, 0, sizeof(unsigned int), s) != cudaSuccess) return MTP_ERR_CUDA;
        j.draw_i = i;
        j.base0 = static_cast<const char*>(dft_logits) + (size_t)i * V * esz;
        if (launch_sample(j, sms, s) != cudaSuccess) return MTP_ERR_CUDA;
    }
    return MTP_OK;
}

int mtp_last_error(const void* ws, mtp_stream_t stream) {
    if (!ws) return MTP_ERR_WORKSPACE;
    int st = 0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const WsHeader* h = static_cast<const WsHeader*>(ws);
    if (cudaMemcpyAsync(&st, &h->status, sizeof st, cudaMemcpyDeviceToHost, s) != cudaSuccess) return MTP_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MTP_ERR_CUDA;
    return st;
}

const char* mtp_strerror(int code) {
    switch (code) {
    case MTP_OK: return "ok";
    case MTP_ERR_ARG: return "invalid argument";
    case MTP_ERR_UNSUPPORTED: return "unsupported size, layout or dtype";
    case MTP_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case MTP_ERR_CUDA: return "CUDA launch or copy failed";
    case MTP_ERR_TIMEOUT: return "grid barrier timed out";
    case MTP_ERR_CAPACITY: return "sampling candidate set exceeded its capacity";
    default: return "unknown error";
    }
}

int mtp_debug_barrier_timeout(void* ws, size_t ws_bytes, int timeout_us, mtp_stream_t stream) {
    if (check_workspace(ws, ws_bytes, sizeof(WsHeader)) != MTP_OK) return MTP_ERR_WORKSPACE;
    if (timeout_us < 1 || timeout_us > 1000000) return MTP_ERR_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(ws, 0, sizeof(WsHeader), s) != cudaSuccess) return MTP_ERR_CUDA;
    cudaError_t e = launch_barrier_timeout_probe(static_cast<WsHeader*>(ws), 1000ull * (unsigned)timeout_us, s);
    return e == cudaSuccess ? MTP_OK : MTP_ERR_CUDA;
}

}  // extern "C"
