// draft_kernel.cuh -- the persistent draft-block kernel.
//
// One cooperative launch runs all N draft steps of all B sequences ("Fused
// NextN draft graph": one launch + one readback; the token -> embedding ->
// hidden-state chain never leaves the device).  Each step is a fixed
// sequence of phases separated by grid barriers ("Gemma 4 MTP", sec. 4):
//
//   PRE     e = E[tok] * s;  x = W_pre [rms(e); rms(h)]
//   per block l:
//     Q     x_l (residual update of the previous block), q = W_q rms(x_l)
//     ATT   q-norm + RoPE, split-K cross-attention into the target KV view
//           (sec. 5: read-only, one mask for every step), last-arriver merge
//     O     y = W_o o
//     FFN1  x_m = x_l + rms(y);  m = gelu_tanh(W_g rms(x_m)) * (W_u rms(x_m))
//     FFN2  y2 = W_d m
//   POST    h = W_post rms(x_m + rms(y2))
//   HEAD    z = E h (softcap), packed-key argmax folded across the grid
//
// Norms and residual updates run redundantly in every CTA's phase prologue
// (each CTA needs the whole input vector of its GEMV anyway), so they cost no
// barrier.  Weights stream through 16-byte no-L1-allocate loads, one warp per
// output row; activations are fp32 in shared memory.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "draft.cuh"

namespace mtp {

// ---------------------------------------------------------------------------
// weight chunk unpacking: 16 bytes -> EPC fp32 values
// ---------------------------------------------------------------------------
template <typename WT> struct Chunk;
template <> struct Chunk<uint16_t> {
    static constexpr int EPC = 8;
    static __device__ __forceinline__ float dot(const uint4& w, const float* a) {
        const float4 a0 = *reinterpret_cast<const float4*>(a);
        const float4 a1 = *reinterpret_cast<const float4*>(a + 4);
        float s = bf16_lo(w.x) * a0.x;
        s = fmaf(bf16_hi(w.x), a0.y, s);
        s = fmaf(bf16_lo(w.y), a0.z, s);
        s = fmaf(bf16_hi(w.y), a0.w, s);
        s = fmaf(bf16_lo(w.z), a1.x, s);
        s = fmaf(bf16_hi(w.z), a1.y, s);
        s = fmaf(bf16_lo(w.w), a1.z, s);
        s = fmaf(bf16_hi(w.w), a1.w, s);
        return s;
    }
};
template <> struct Chunk<float> {
    static constexpr int EPC = 4;
    static __device__ __forceinline__ float dot(const uint4& w, const float* a) {
        const float4 a0 = *reinterpret_cast<const float4*>(a);
        float s = __uint_as_float(w.x) * a0.x;
        s = fmaf(__uint_as_float(w.y), a0.y, s);
        s = fmaf(__uint_as_float(w.z), a0.z, s);
        s = fmaf(__uint_as_float(w.w), a0.w, s);
        return s;
    }
};

// ---------------------------------------------------------------------------
// GEMV over a row range: out[r, b] = sum_c W[r, c] act[b, c] for b in
// [b0, b0 + NB) (masked by nb), one warp per row, grid-strided over rows.
// TWO = true also computes the same row of a second matrix W2 (GeGLU gate/up).
// ---------------------------------------------------------------------------
template <typename WT, int U, int NB, bool TWO, class Epi>
__device__ __forceinline__ void gemv_rows(const WT* __restrict__ W, const WT* __restrict__ W2, int rows, int K,
                                          const float* act, int lda, int b0, int nb, Epi& epi) {
    constexpr int EPC = Chunk<WT>::EPC;
    const int nch = K / EPC;
    const int lane = threadIdx.x & 31;
    const int gw = blockIdx.x * kWarps + (threadIdx.x >> 5);
    const int nw = gridDim.x * kWarps;
    for (int r = gw; r < rows; r += nw) {
        const uint4* wr = reinterpret_cast<const uint4*>(W + (long long)r * K);
        const uint4* wr2 = TWO ? reinterpret_cast<const uint4*>(W2 + (long long)r * K) : nullptr;
        float acc[NB], acc2[NB];
#pragma unroll
        for (int j = 0; j < NB; ++j) { acc[j] = 0.f; acc2[j] = 0.f; }
        for (int c0 = 0; c0 < nch; c0 += 32 * U) {
            uint4 w[U], w2[TWO ? U : 1];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + lane + 32 * u;
                w[u] = c < nch ? ld_stream16(wr + c) : make_uint4(0u, 0u, 0u, 0u);
                if (TWO) w2[u] = c < nch ? ld_stream16(wr2 + c) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + lane + 32 * u;
                if (c < nch) {
#pragma unroll
                    for (int j = 0; j < NB; ++j) {
                        if (b0 + j < nb) {
                            const float* a = act + (long long)(b0 + j) * lda + c * EPC;
                            acc[j] += Chunk<WT>::dot(w[u], a);
                            if (TWO) acc2[j] += Chunk<WT>::dot(w2[u], a);
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int j = 0; j < NB; ++j) {
            acc[j] = warp_sum(acc[j]);
            if (TWO) acc2[j] = warp_sum(acc2[j]);
        }
        epi.apply(r, b0, nb, acc, acc2);
    }
}

template <typename WT, int U, bool TWO, class Epi>
__device__ __forceinline__ void gemv(const WT* W, const WT* W2, int rows, int K, const float* act, int lda, int nb,
                                     Epi& epi) {
    if (nb == 1) {
        gemv_rows<WT, U, 1, TWO>(W, W2, rows, K, act, lda, 0, 1, epi);
    } else {
        for (int b0 = 0; b0 < nb; b0 += 4) gemv_rows<WT, U, 4, TWO>(W, W2, rows, K, act, lda, b0, nb, epi);
    }
}

// out[b * ldo + r] = v
struct StoreEpi {
    float* out;
    int ldo;
    template <int NB>
    __device__ __forceinline__ void apply(int r, int b0, int nb, const float (&acc)[NB], const float (&)[NB]) {
        const int lane = threadIdx.x & 31;
#pragma unroll
        for (int j = 0; j < NB; ++j)
            if (lane == j && b0 + j < nb) out[(long long)(b0 + j) * ldo + r] = acc[j];
    }
};

__device__ __forceinline__ float gelu_tanh(float x) {
    const float k0 = 0.7978845608028654f;  // sqrt(2 / pi)
    return 0.5f * x * (1.f + tanhf(k0 * (x + 0.044715f * x * x * x)));
}

// m[b * ldo + r] = gelu_tanh(gate) * up
struct GegluEpi {
    float* out;
    int ldo;
    template <int NB>
    __device__ __forceinline__ void apply(int r, int b0, int nb, const float (&g)[NB], const float (&u)[NB]) {
        const int lane = threadIdx.x & 31;
#pragma unroll
        for (int j = 0; j < NB; ++j)
            if (lane == j && b0 + j < nb) out[(long long)(b0 + j) * ldo + r] = gelu_tanh(g[j]) * u[j];
    }
};

// LM head: softcap, optional logits store, running packed argmax per column
// (lane c & 31 owns column c; two registers cover 64 columns).
struct HeadEpi {
    float* logits;  // [B, N, V] or null
    int V, N, step;
    float softcap;
    unsigned long long best_lo, best_hi;
    template <int NB>
    __device__ __forceinline__ void apply(int r, int b0, int nb, const float (&acc)[NB], const float (&)[NB]) {
        const int lane = threadIdx.x & 31;
#pragma unroll
        for (int j = 0; j < NB; ++j) {
            const int col = b0 + j;
            if (col < nb && lane == (col & 31)) {
                float z = acc[j];
                if (softcap > 0.f) z = softcap * tanhf(z / softcap);
                if (logits) logits[((long long)col * N + step) * V + r] = z;
                const unsigned long long k = pack_argmax(z, (uint32_t)r);
                if (col < 32) best_lo = k > best_lo ? k : best_lo;
                else best_hi = k > best_hi ? k : best_hi;
            }
        }
    }
};

// ---------------------------------------------------------------------------
// prologues: build one sequence's GEMV input vector
// ---------------------------------------------------------------------------

// dst[i] = src[i] * rsqrt(mean(src^2) + eps) * g[i]; src may alias dst.
// All threads of the CTA participate.
__device__ __forceinline__ void rms_into(const float* src, const float* g, int n, float eps, float* dst, float* red) {
    float ss = 0.f;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const float v = src[i];
        ss = fmaf(v, v, ss);
    }
    ss = block_sum(ss, red);
    const float r = 1.0f / sqrtf(ss / (float)n + eps);
    for (int i = threadIdx.x; i < n; i += blockDim.x) dst[i] = src[i] * r * __ldg(g + i);
    __syncthreads();
}

// token consumed by sequence b at step k
__device__ __forceinline__ int step_token(const DraftParams& p, int b, int k) {
    if (k == 0) return p.last_tok[b];
    const uint32_t t = unpack_index(__ldcg(p.amax + (long long)(k - 1) * p.B + b));
    return t < (uint32_t)p.V ? (int)t : 0;   // every slot holds a row index after its HEAD phase
}

enum Phase { PH_PRE, PH_Q, PH_O, PH_FFN1, PH_FFN2, PH_POST, PH_HEAD };

// Writes sequence b's input vector for `phase` into dst (length phase_k).
// `writer` marks the one CTA that also stores residual-stream updates.
template <typename WT>
__device__ void build_act(const DraftParams& p, int phase, int k, int l, int b, float* dst, float* tmp, bool writer,
                          float* red) {
    switch (phase) {
    case PH_PRE: {
        const int tok = step_token(p, b, k);
        const WT* er = reinterpret_cast<const WT*>(p.tok_embd) + (long long)tok * p.d_t;
        for (int i = threadIdx.x; i < p.d_t; i += blockDim.x) dst[i] = ld_elem<WT>(er, i) * p.emb_scale;
        const float* h = k == 0 ? p.h_prev + (long long)b * p.d_t : p.HN + (long long)b * p.d_t;
        for (int i = threadIdx.x; i < p.d_t; i += blockDim.x) dst[p.d_t + i] = __ldcg(h + i);
        __syncthreads();
        rms_into(dst, p.norm_e, p.d_t, p.eps, dst, red);
        rms_into(dst + p.d_t, p.norm_h, p.d_t, p.eps, dst + p.d_t, red);
        break;
    }
    case PH_Q: {
        const int n = p.d_a;
        if (l == 0) {
            for (int i = threadIdx.x; i < n; i += blockDim.x) tmp[i] = __ldcg(p.XB + (long long)b * n + i);
            __syncthreads();
        } else {
            for (int i = threadIdx.x; i < n; i += blockDim.x) {
                dst[i] = __ldcg(p.Y2 + (long long)b * n + i);
                tmp[i] = __ldcg(p.XM + (long long)b * n + i);
            }
            __syncthreads();
            rms_into(dst, p.blk[l - 1].post_ffn_norm, n, p.eps, dst, red);
            for (int i = threadIdx.x; i < n; i += blockDim.x) {
                const float x = tmp[i] + dst[i];
                tmp[i] = x;
                if (writer) p.XB[(long long)b * n + i] = x;
            }
            __syncthreads();
        }
        rms_into(tmp, p.blk[l].attn_norm, n, p.eps, dst, red);
        break;
    }
    case PH_FFN1: {
        const int n = p.d_a;
        for (int i = threadIdx.x; i < n; i += blockDim.x) {
            dst[i] = __ldcg(p.YB + (long long)b * n + i);
            tmp[i] = __ldcg(p.XB + (long long)b * n + i);
        }
        __syncthreads();
        rms_into(dst, p.blk[l].post_attn_norm, n, p.eps, dst, red);
        for (int i = threadIdx.x; i < n; i += blockDim.x) {
            const float x = tmp[i] + dst[i];
            tmp[i] = x;
            if (writer) p.XM[(long long)b * n + i] = x;
        }
        __syncthreads();
        rms_into(tmp, p.blk[l].pre_ffn_norm, n, p.eps, dst, red);
        break;
    }
    case PH_POST: {
        const int n = p.d_a;
        for (int i = threadIdx.x; i < n; i += blockDim.x) {
            dst[i] = __ldcg(p.Y2 + (long long)b * n + i);
            tmp[i] = __ldcg(p.XM + (long long)b * n + i);
        }
        __syncthreads();
        rms_into(dst, p.blk[p.L - 1].post_ffn_norm, n, p.eps, dst, red);
        for (int i = threadIdx.x; i < n; i += blockDim.x) tmp[i] += dst[i];
        __syncthreads();
        rms_into(tmp, p.final_norm, n, p.eps, dst, red);
        break;
    }
    case PH_O: {
        const int n = p.Hq * p.hd;
        for (int i = threadIdx.x; i < n; i += blockDim.x) dst[i] = __ldcg(p.OB + (long long)b * n + i);
        __syncthreads();
        break;
    }
    case PH_FFN2: {
        const int n = p.F;
        for (int i = threadIdx.x; i < n; i += blockDim.x) dst[i] = __ldcg(p.MB + (long long)b * n + i);
        __syncthreads();
        break;
    }
    case PH_HEAD: {
        const int n = p.d_t;
        for (int i = threadIdx.x; i < n; i += blockDim.x) dst[i] = __ldcg(p.HN + (long long)b * n + i);
        __syncthreads();
        break;
    }
    }
}

__device__ __forceinline__ int phase_k(const DraftParams& p, int phase) {
    switch (phase) {
    case PH_PRE: return 2 * p.d_t;
    case PH_Q: case PH_FFN1: case PH_POST: return p.d_a;
    case PH_O: return p.Hq * p.hd;
    case PH_FFN2: return p.F;
    default: return p.d_t;
    }
}

// Stage the inputs of a GEMV phase.  Shared-memory mode: every CTA builds all
// B vectors into `smem_act` (stride K) and no barrier is needed.  Global mode:
// CTA c builds sequences b = c, c + grid, ... into p.ACT and a barrier
// follows.  Returns the activation pointer and stride, or null if a barrier
// failed.
template <typename WT>
__device__ const float* stage_act(const DraftParams& p, int phase, int k, int l, float* smem_act, float* smem_tmp,
                                  float* red, unsigned int& epoch, int& lda, bool& ok) {
    const int K = phase_k(p, phase);
    ok = true;
    if (p.act_smem) {
        for (int b = 0; b < p.B; ++b)
            build_act<WT>(p, phase, k, l, b, smem_act + (long long)b * K, smem_tmp, blockIdx.x == 0, red);
        lda = K;
        return smem_act;
    }
    // global mode: copy-only inputs are read in place
    if (phase == PH_O) { lda = K; return p.OB; }
    if (phase == PH_FFN2) { lda = K; return p.MB; }
    if (phase == PH_HEAD) { lda = K; return p.HN; }
    for (int b = blockIdx.x; b < p.B; b += gridDim.x) {
        build_act<WT>(p, phase, k, l, b, smem_act, smem_tmp, true, red);
        for (int i = threadIdx.x; i < K; i += blockDim.x) p.ACT[(long long)b * p.kmax + i] = smem_act[i];
        __syncthreads();
    }
    ok = grid_barrier(p.hdr, epoch, p.timeout_ns, gridDim.x);
    lda = p.kmax;
    return p.ACT;
}

// ---------------------------------------------------------------------------
// attention (split-K over key ranges, online softmax, last-arriver merge)
// ---------------------------------------------------------------------------

__device__ __forceinline__ int view_lo(const KView& v, int kv_len) {
    return (v.window > 0 && kv_len > v.window) ? kv_len - v.window : 0;
}

template <typename WT, int HD>
__device__ void attention_phase(const DraftParams& p, int l, int k, unsigned char* smem) {
    constexpr int CK = attn_keys(HD, (int)sizeof(WT));      // keys per staged sub-chunk
    constexpr int ROWB = HD * (int)sizeof(WT) + kAttnPad;   // bytes per staged row
    constexpr int BUFB = 2 * CK * ROWB;                     // one K + V sub-chunk
    constexpr int NCP = (2 * CK * (HD * (int)sizeof(WT) / 16) + kThreads - 1) / kThreads;  // copies per thread
    constexpr int CPR = HD * (int)sizeof(WT) / 16;          // 16-byte chunks per row
    constexpr int EPC = 16 / (int)sizeof(WT);
    const KView& vw = p.views[p.blk[l].view];
    const int grp = p.Hq / p.Hkv;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    double* invf = reinterpret_cast<double*>(smem);     // [HD/2] RoPE inverse frequencies
    float* qs = reinterpret_cast<float*>(invf + HD / 2);  // [grp][HD]
    float* os = qs + grp * HD;                           // [grp][HD]
    float* sc = os + grp * HD;                           // [grp][CK]
    float* mrow = sc + grp * CK;                         // [grp]
    float* lrow = mrow + 16;                             // [grp]
    float* arow = lrow + 16;                             // [grp]
    unsigned char* kvbuf = reinterpret_cast<unsigned char*>(arow + 16);  // 2 x (K rows, V rows)
    __shared__ int s_last;

    // RoPE inverse frequencies, once per phase (fp64 is scarce on this part)
    {
        const double ltheta = log((double)vw.theta);
        for (int i = tid; i < HD / 2; i += blockDim.x) invf[i] = exp(-2.0 * (double)i / (double)HD * ltheta);
        __syncthreads();
    }
    long long total = 0;
    for (int b = 0; b < p.B; ++b) total += (long long)(p.kv_len[b] - view_lo(vw, p.kv_len[b])) * p.Hkv;
    // keys per item: about one item per CTA (two when every CTA would get
    // more than 512 keys, to even out ragged sequence lengths)
    const long long target = (total / gridDim.x <= 512) ? gridDim.x : 2LL * gridDim.x;
    long long kpi = (total + target - 1) / target;
    kpi = ((kpi + CK - 1) / CK) * CK;
    if (kpi < CK) kpi = CK;
    long long n_items = 0;
    for (int b = 0; b < p.B; ++b) {
        const long long n = p.kv_len[b] - view_lo(vw, p.kv_len[b]);
        n_items += p.Hkv * ((n + kpi - 1) / kpi);
    }
    const int PSZ = grp * (HD + 2);  // floats per partial: m[grp], l[grp], o[grp][HD]

    for (long long it = blockIdx.x; it < n_items; it += gridDim.x) {
        // item -> (b, g, s)
        int b = 0;
        long long base = 0, S = 1;
        for (b = 0; b < p.B; ++b) {
            const long long n = p.kv_len[b] - view_lo(vw, p.kv_len[b]);
            S = (n + kpi - 1) / kpi;
            if (it < base + p.Hkv * S) break;
            base += p.Hkv * S;
        }
        const int g = (int)((it - base) / S);
        const int s = (int)((it - base) % S);
        const long long bg_base = base + (long long)g * S;
        const int kv_len = p.kv_len[b];
        const int lo = view_lo(vw, kv_len);
        const long long t_beg = lo + (long long)s * kpi;
        const long long t_end = (t_beg + kpi < kv_len) ? t_beg + kpi : kv_len;

        // K/V sub-chunks of CK keys go to shared memory through cp.async, two
        // buffers deep: sub-chunk i + 1 is in flight while i is used.  Rows
        // past the range are zero-filled so they never carry NaN.
        const WT* kbase = reinterpret_cast<const WT*>(vw.k) + (long long)b * vw.sb + (long long)g * vw.sh;
        const WT* vbase = reinterpret_cast<const WT*>(vw.v) + (long long)b * vw.sb + (long long)g * vw.sh;
        const int nsub = (int)((t_end - t_beg + CK - 1) / CK);
        auto stage = [&](int i) {
            const long long t0 = t_beg + (long long)i * CK;
            const int cnt = (int)((t_end - t0) < CK ? (t_end - t0) : CK);
            const int s0 = (int)(t0 % vw.cap);
            unsigned char* buf = kvbuf + (i & 1) * BUFB;
#pragma unroll
            for (int u = 0; u < NCP; ++u) {
                const int c = tid + u * kThreads;
                if (c < 2 * CK * CPR) {
                    const int which = c / (CK * CPR);
                    const int j = (c / CPR) % CK;
                    const int q = c % CPR;
                    unsigned char* dst = buf + which * CK * ROWB + j * ROWB + q * 16;
                    if (j < cnt) {
                        int slot = s0 + j;
                        if (slot >= vw.cap) slot %= vw.cap;
                        cp_async16(dst, (which ? vbase : kbase) + (long long)slot * vw.st + q * EPC);
                    } else {
                        *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
            }
            cp_async_commit();
        };
        stage(0);

        // q-norm + RoPE for the group's heads (warp h handles head h), scaled by attn_scale
        if (warp < grp) {
            const int h = g * grp + warp;
            const float* qraw = p.QR + (long long)b * p.Hq * HD + (long long)h * HD;
            float ss = 0.f;
            for (int d = lane; d < HD; d += 32) {
                const float v = __ldcg(qraw + d);
                qs[warp * HD + d] = v;
                ss = fmaf(v, v, ss);
            }
            ss = warp_sum(ss);
            const float r = 1.0f / sqrtf(ss / (float)HD + p.eps);
            const float* gq = p.blk[l].q_norm;
            __syncwarp();
            const double pos = (double)kv_len + (double)k;
            constexpr int PPL = HD / 64 > 0 ? HD / 64 : 1;  // rotation pairs per lane
            float ra[PPL], rb[PPL];
#pragma unroll
            for (int m = 0; m < PPL; ++m) {
                const int i = lane + 32 * m;
                if (i < HD / 2) {
                    const float a = qs[warp * HD + i] * r * __ldg(gq + i);
                    const float c = qs[warp * HD + i + HD / 2] * r * __ldg(gq + i + HD / 2);
                    // angle pos * theta^(-2i/HD) in fp64, reduced to [-pi, pi] before the fp32 sin/cos
                    double ang = pos * invf[i];
                    ang -= 6.283185307179586 * rint(ang * 0.15915494309189535);
                    float sn, cs;
                    sincosf((float)ang, &sn, &cs);
                    ra[m] = (a * cs - c * sn) * p.attn_scale;
                    rb[m] = (a * sn + c * cs) * p.attn_scale;
                }
            }
            __syncwarp();
#pragma unroll
            for (int m = 0; m < PPL; ++m) {
                const int i = lane + 32 * m;
                if (i < HD / 2) {
                    qs[warp * HD + i] = ra[m];
                    qs[warp * HD + i + HD / 2] = rb[m];
                }
            }
            if (lane == 0) { mrow[warp] = -INFINITY; lrow[warp] = 0.f; }
        }
        for (int o = tid; o < grp * HD; o += blockDim.x) os[o] = 0.f;
        __syncthreads();

        for (int i = 0; i < nsub; ++i) {
            const long long t0 = t_beg + (long long)i * CK;
            const int cnt = (int)((t_end - t0) < CK ? (t_end - t0) : CK);
            if (i + 1 < nsub) {
                stage(i + 1);
                cp_async_wait<1>();
            } else {
                cp_async_wait<0>();
            }
            __syncthreads();
            const unsigned char* ks = kvbuf + (i & 1) * BUFB;
            const unsigned char* vs = ks + CK * ROWB;
            // scores
            for (int pr = tid; pr < grp * CK; pr += blockDim.x) {
                const int h = pr / CK, j = pr % CK;
                float sv = -INFINITY;
                if (j < cnt) {
                    const float* qh = qs + h * HD;
                    const unsigned char* kr = ks + j * ROWB;
                    float acc = 0.f;
#pragma unroll 4
                    for (int q = 0; q < CPR; ++q) {
                        const uint4 w = *reinterpret_cast<const uint4*>(kr + q * 16);
                        acc += Chunk<WT>::dot(w, qh + q * EPC);
                    }
                    sv = acc;
                }
                sc[h * CK + j] = sv;
            }
            __syncthreads();
            // online softmax update (warp h owns head h)
            if (warp < grp) {
                float mx = -INFINITY;
                for (int j = lane; j < CK; j += 32) mx = fmaxf(mx, sc[warp * CK + j]);
                mx = warp_max(mx);
                const float m_old = mrow[warp];
                const float m_new = fmaxf(m_old, mx);
                const float alpha = expf(m_old - m_new);
                float ls = 0.f;
                for (int j = lane; j < CK; j += 32) {
                    const float e = j < cnt ? expf(sc[warp * CK + j] - m_new) : 0.f;
                    sc[warp * CK + j] = e;
                    ls += e;
                }
                ls = warp_sum(ls);
                __syncwarp();
                if (lane == 0) {
                    mrow[warp] = m_new;
                    lrow[warp] = lrow[warp] * alpha + ls;
                    arow[warp] = alpha;
                }
            }
            __syncthreads();
            // o = o * alpha + P V
            for (int o = tid; o < grp * HD; o += blockDim.x) {
                const int h = o / HD, d = o % HD;
                float acc = os[o] * arow[h];
                const float* ph = sc + h * CK;
                for (int j = 0; j < cnt; ++j) {
                    const WT* vr = reinterpret_cast<const WT*>(vs + j * ROWB);
                    float vv;
                    if (sizeof(WT) == 2) vv = bf16_to_f32(reinterpret_cast<const uint16_t*>(vr)[d]);
                    else vv = reinterpret_cast<const float*>(vr)[d];
                    acc = fmaf(ph[j], vv, acc);
                }
                os[o] = acc;
            }
            __syncthreads();
        }

        // partial (m, l, o) of this item
        float* part = p.PART + it * PSZ;
        for (int h = tid; h < grp; h += blockDim.x) { part[h] = mrow[h]; part[grp + h] = lrow[h]; }
        for (int o = tid; o < grp * HD; o += blockDim.x) part[2 * grp + o] = os[o];
        __threadfence();
        __syncthreads();
        if (tid == 0) s_last = (atomicAdd(p.att_cnt + b * p.Hkv + g, 1u) == (unsigned)(S - 1));
        __syncthreads();
        if (s_last) {
            __threadfence();
            // merge the S partials of (b, g) into OB[b, g*grp .. (g+1)*grp):
            // warp h finds head h's max and weights with its lanes spread over
            // the partials; then every output sums the S weighted partials
            // with independent loads in flight
            float* M = mrow;   // reuse: per-head max and total
            float* Lt = lrow;
            float* es = reinterpret_cast<float*>(kvbuf);   // [S][grp] merge weights (K/V stage is free now)
            const bool cached = S * grp <= (long long)(BUFB / sizeof(float));
            if (warp < grp) {
                const int h = warp;
                float mm = -INFINITY;
                for (long long q = lane; q < S; q += 32) mm = fmaxf(mm, __ldcg(p.PART + (bg_base + q) * PSZ + h));
                mm = warp_max(mm);
                float lt = 0.f;
                for (long long q = lane; q < S; q += 32) {
                    const float* pq = p.PART + (bg_base + q) * PSZ;
                    const float e = expf(__ldcg(pq + h) - mm);
                    if (cached) es[q * grp + h] = e;
                    lt += e * __ldcg(pq + grp + h);
                }
                lt = warp_sum(lt);
                if (lane == 0) {
                    M[h] = mm;
                    Lt[h] = lt;
                }
            }
            __syncthreads();
            for (int o = tid; o < grp * HD; o += blockDim.x) {
                const int h = o / HD;
                float acc = 0.f;
                long long q = 0;
                for (; q + 4 <= S; q += 4) {
                    float v[4], e[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const float* pq = p.PART + (bg_base + q + u) * PSZ;
                        v[u] = __ldcg(pq + 2 * grp + o);
                        e[u] = cached ? es[(q + u) * grp + h] : expf(__ldcg(pq + h) - M[h]);
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u) acc = fmaf(e[u], v[u], acc);
                }
                for (; q < S; ++q) {
                    const float* pq = p.PART + (bg_base + q) * PSZ;
                    const float e = cached ? es[q * grp + h] : expf(__ldcg(pq + h) - M[h]);
                    acc = fmaf(e, __ldcg(pq + 2 * grp + o), acc);
                }
                p.OB[(long long)b * p.Hq * HD + (long long)g * grp * HD + o] = acc / Lt[h];
            }
            if (tid == 0) p.att_cnt[b * p.Hkv + g] = 0u;
            __syncthreads();
        }
    }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <typename WT, int HD>
__global__ void __launch_bounds__(kThreads, 1) draft_kernel(const __grid_constant__ DraftParams p) {
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ float red[kWarps];
    __shared__ unsigned long long head_best[kWarps][32];
    unsigned int epoch = 0;
    float* tmp = reinterpret_cast<float*>(smem);                 // [max(d_a)] residual scratch
    float* act = tmp + ((p.d_a + 3) & ~3);                       // activations
    constexpr int U = 8;
    bool ok = true;
    int lda = 0;

    // device-side input checks: every CTA evaluates the same predicate, so on
    // bad inputs all CTAs return before the first barrier
    {
        bool bad = false;
        for (int b = 0; b < p.B; ++b) {
            const int kl = p.kv_len[b], tk = p.last_tok[b];
            if (kl < 1 || tk < 0 || tk >= p.V) bad = true;
            for (int l = 0; l < p.L; ++l) {
                const KView& v = p.views[p.blk[l].view];
                if (v.window == 0 && kl > v.cap) bad = true;
            }
        }
        if (bad) {
            if (blockIdx.x == 0 && threadIdx.x == 0) atomicCAS(&p.hdr->status, 0, MTP_ERR_ARG);
            return;
        }
    }
    // zero the argmax slots of every step (first read after >= 1 barrier)
    if (blockIdx.x == 0)
        for (int i = threadIdx.x; i < p.N * p.B; i += blockDim.x) p.amax[i] = 0ull;

    for (int k = 0; k < p.N; ++k) {
        // ---- PRE ----
        if (blockIdx.x == 0 && k > 0)
            for (int b = threadIdx.x; b < p.B; b += blockDim.x)
                p.out_drafts[(long long)b * p.N + (k - 1)] = step_token(p, b, k);
        {
            const float* a = stage_act<WT>(p, PH_PRE, k, 0, act, tmp, red, epoch, lda, ok);
            if (!ok) return;
            StoreEpi e{p.XB, p.d_a};
            gemv<WT, U, false>(reinterpret_cast<const WT*>(p.w_pre), nullptr, p.d_a, 2 * p.d_t, a, lda, p.B, e);
        }
        if (!grid_barrier(p.hdr, epoch, p.timeout_ns, gridDim.x)) return;

        for (int l = 0; l < p.L; ++l) {
            const BlkW& bw = p.blk[l];
            // ---- Q ----
            {
                const float* a = stage_act<WT>(p, PH_Q, k, l, act, tmp, red, epoch, lda, ok);
                if (!ok) return;
                StoreEpi e{p.QR, p.Hq * p.hd};
                gemv<WT, U, false>(reinterpret_cast<const WT*>(bw.w_q), nullptr, p.Hq * p.hd, p.d_a, a, lda, p.B, e);
            }
            if (!grid_barrier(p.hdr, epoch, p.timeout_ns, gridDim.x)) return;
            // ---- ATT ----
            attention_phase<WT, HD>(p, l, k, smem);
            if (!grid_barrier(p.hdr, epoch, p.timeout_ns, gridDim.x)) return;
            // ---- O ----
            {
                const float* a = stage_act<WT>(p, PH_O, k, l, act, tmp, red, epoch, lda, ok);
                if (!ok) return;
                StoreEpi e{p.YB, p.d_a};
                gemv<WT, U, false>(reinterpret_cast<const WT*>(bw.w_o), nullptr, p.d_a, p.Hq * p.hd, a, lda, p.B, e);
            }
            if (!grid_barrier(p.hdr, epoch, p.timeout_ns, gridDim.x)) return;
            // ---- FFN1 (gate and up share the input; GeGLU in the epilogue) ----
            {
                const float* a = stage_act<WT>(p, PH_FFN1, k, l, act, tmp, red, epoch, lda, ok);
                if (!ok) return;
                GegluEpi e{p.MB, p.F};
                gemv<WT, U / 2, true>(reinterpret_cast<const WT*>(bw.w_gate), reinterpret_cast<const WT*>(bw.w_up),
                                      p.F, p.d_a, a, lda, p.B, e);
            }
            if (!grid_barrier(p.hdr, epoch, p.timeout_ns, gridDim.x)) return;
            // ---- FFN2 ----
            {
                const float* a = stage_act<WT>(p, PH_FFN2, k, l, act, tmp, red, epoch, lda, ok);
                if (!ok) return;
                StoreEpi e{p.Y2, p.d_a};
                gemv<WT, U, false>(reinterpret_cast<const WT*>(bw.w_down), nullptr, p.d_a, p.F, a, lda, p.B, e);
            }
            if (!grid_barrier(p.hdr, epoch, p.timeout_ns, gridDim.x)) return;
        }
        // ---- POST ----
        {
            const float* a = stage_act<WT>(p, PH_POST, k, 0, act, tmp, red, epoch, lda, ok);
            if (!ok) return;
            StoreEpi e{p.HN, p.d_t};
            gemv<WT, U, false>(reinterpret_cast<const WT*>(p.w_post), nullptr, p.d_t, p.d_a, a, lda, p.B, e);
        }
        if (!grid_barrier(p.hdr, epoch, p.timeout_ns, gridDim.x)) return;
        // ---- HEAD ----
        {
            const float* a = stage_act<WT>(p, PH_HEAD, k, 0, act, tmp, red, epoch, lda, ok);
            if (!ok) return;
            HeadEpi e{p.out_logits, p.V, p.N, k, p.softcap, 0ull, 0ull};
            gemv<WT, U, false>(reinterpret_cast<const WT*>(p.tok_embd), nullptr, p.V, p.d_t, a, lda, p.B, e);
            // fold the per-lane bests: per CTA in shared memory, one atomic per column
            const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
            for (int c0 = 0; c0 < p.B; c0 += 32) {
                head_best[warp][lane] = c0 == 0 ? e.best_lo : e.best_hi;   // column c0 + lane
                __syncthreads();
                if (threadIdx.x < 32 && c0 + (int)threadIdx.x < p.B) {
                    unsigned long long m = 0ull;
                    for (int w = 0; w < kWarps; ++w) m = head_best[w][threadIdx.x] > m ? head_best[w][threadIdx.x] : m;
                    atomicMax(p.amax + (long long)k * p.B + c0 + threadIdx.x, m);
                }
                __syncthreads();
            }
        }
        if (!grid_barrier(p.hdr, epoch, p.timeout_ns, gridDim.x)) return;
    }
    // outputs of the last step
    if (blockIdx.x == 0) {
        for (int b = threadIdx.x; b < p.B; b += blockDim.x)
            p.out_drafts[(long long)b * p.N + (p.N - 1)] = step_token(p, b, p.N);
        if (p.out_h_last)
            for (long long i = threadIdx.x; i < (long long)p.B * p.d_t; i += blockDim.x) p.out_h_last[i] = __ldcg(p.HN + i);
    }
}

template <typename WT, int HD>
cudaError_t launch_draft_t(const DraftParams& p, int grid, size_t smem, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(draft_kernel<WT, HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    void* args[] = {const_cast<DraftParams*>(&p)};
    return cudaLaunchCooperativeKernel((const void*)draft_kernel<WT, HD>, dim3(grid), dim3(kThreads), args, smem, s);
}

template <typename WT, int HD>
int draft_blocks_per_sm_t(size_t smem) {
    int n = 0;
    cudaFuncSetAttribute(draft_kernel<WT, HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, draft_kernel<WT, HD>, kThreads, smem) != cudaSuccess) return 0;
    return n;
}

}  // namespace mtp
