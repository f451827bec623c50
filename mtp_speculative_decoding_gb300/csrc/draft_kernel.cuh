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
// The dense NextN drafter ("MTP decoding (--mtp)", "Requirements"; its own
// block and KV) runs through the same kernel (nextn = 1, one block at the
// backbone width): PRE is eh_proj; Q is the fused query / key / value
// projection, after which each (sequence, KV head) key is normed, rotated and
// stored with its value in the drafter's KV before the causal attention
// reads it; FFN1 adds the attention output without a norm and gates with
// SiLU; POST is no projection: h' = x_m + y2 (the next step's hidden state)
// and the head's input is head_norm(h').  Catch-up rows (the accepted drafts
// with the target's hidden states) run as iterations k < 0 of PRE and the
// key / value rows of Q only.
//
// Norms and residual updates run redundantly in every CTA's phase prologue
// (each CTA needs the whole input vector of its GEMV anyway), so they cost no
// barrier.  At one sequence (and with fp32, Q8_0 or centroid-routed models)
// the weights stream through 16-byte no-L1-allocate loads under an L2
// evict-first policy, a warp per output row (at one sequence: two warps per
// row when rows are few, two rows per warp when rows are short); from two
// sequences the LM head, and the projections once their inputs no longer fit
// in shared memory, run on the tensor cores (tc_head, tc_gemm).  Activations
// are fp32.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include <cuda_bf16.h>

#include "common.cuh"
#include "draft.cuh"
#include "sample.cuh"

namespace mtp {

// ---------------------------------------------------------------------------
// weight chunk unpacking: 16 bytes -> EPC fp32 values
// ---------------------------------------------------------------------------
template <typename WT> struct Chunk;
template <> struct Chunk<uint16_t> {
    static constexpr int EPC = 8;
    static constexpr bool QUANT = false;
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
    // dot with 8 values held in registers (constant indices only)
    static __device__ __forceinline__ float dotr(const uint4& w, const float* a) {
        float s = bf16_lo(w.x) * a[0];
        s = fmaf(bf16_hi(w.x), a[1], s);
        s = fmaf(bf16_lo(w.y), a[2], s);
        s = fmaf(bf16_hi(w.y), a[3], s);
        s = fmaf(bf16_lo(w.z), a[4], s);
        s = fmaf(bf16_hi(w.z), a[5], s);
        s = fmaf(bf16_lo(w.w), a[6], s);
        s = fmaf(bf16_hi(w.w), a[7], s);
        return s;
    }
    static __device__ __forceinline__ float elem(const uint4& w, int e) {
        const uint32_t x = e < 2 ? w.x : e < 4 ? w.y : e < 6 ? w.z : w.w;
        return (e & 1) ? bf16_hi(x) : bf16_lo(x);
    }
};
template <> struct Chunk<float> {
    static constexpr int EPC = 4;
    static constexpr bool QUANT = false;
    static __device__ __forceinline__ float dot(const uint4& w, const float* a) {
        const float4 a0 = *reinterpret_cast<const float4*>(a);
        float s = __uint_as_float(w.x) * a0.x;
        s = fmaf(__uint_as_float(w.y), a0.y, s);
        s = fmaf(__uint_as_float(w.z), a0.z, s);
        s = fmaf(__uint_as_float(w.w), a0.w, s);
        return s;
    }
    static __device__ __forceinline__ float dotr(const uint4& w, const float* a) {
        float s = __uint_as_float(w.x) * a[0];
        s = fmaf(__uint_as_float(w.y), a[1], s);
        s = fmaf(__uint_as_float(w.z), a[2], s);
        s = fmaf(__uint_as_float(w.w), a[3], s);
        return s;
    }
    static __device__ __forceinline__ float elem(const uint4& w, int e) {
        return __uint_as_float(e == 0 ? w.x : e == 1 ? w.y : e == 2 ? w.z : w.w);
    }
};

// Q8_0 codes ("opus-mtp-turbo: Track 1 report", item 3): 16 int8 codes per
// chunk; the weight is the code times its 32-weight block's binary16 scale,
// which the GEMVs apply per chunk (chunk_scale)
template <> struct Chunk<int8_t> {
    static constexpr int EPC = 16;
    static constexpr bool QUANT = true;
    static __device__ __forceinline__ float dot(const uint4& w, const float* a) {
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
        float s = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float4 av = *reinterpret_cast<const float4*>(a + 4 * k);
            s = fmaf((float)(int8_t)(ws[k] & 0xffu), av.x, s);
            s = fmaf((float)(int8_t)((ws[k] >> 8) & 0xffu), av.y, s);
            s = fmaf((float)(int8_t)((ws[k] >> 16) & 0xffu), av.z, s);
            s = fmaf((float)(int8_t)(ws[k] >> 24), av.w, s);
        }
        return s;
    }
};
// Q4_0 codes (the same report's Q4_0 column, ggml's block format): 16 bytes
// per block of 32 weights, byte j holding the code of weight j in its low
// four bits and that of weight j + 16 in its high four; the weight is
// (code - 8) times the block's binary16 scale (chunk_scale).  One chunk is
// one block.
struct Q4Code {
    uint8_t packed;
};
template <> struct Chunk<Q4Code> {
    static constexpr int EPC = 32;
    static constexpr bool QUANT = true;
    static __device__ __forceinline__ float dot(const uint4& w, const float* a) {
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
        float s = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float4 lo = *reinterpret_cast<const float4*>(a + 4 * k);        // weights 4k .. 4k + 3
            const float4 hi = *reinterpret_cast<const float4*>(a + 16 + 4 * k);   // weights 16 + 4k ..
            const uint32_t x = ws[k];
            s = fmaf((float)((int)(x & 15u) - 8), lo.x, s);
            s = fmaf((float)((int)((x >> 8) & 15u) - 8), lo.y, s);
            s = fmaf((float)((int)((x >> 16) & 15u) - 8), lo.z, s);
            s = fmaf((float)((int)((x >> 24) & 15u) - 8), lo.w, s);
            s = fmaf((float)((int)((x >> 4) & 15u) - 8), hi.x, s);
            s = fmaf((float)((int)((x >> 12) & 15u) - 8), hi.y, s);
            s = fmaf((float)((int)((x >> 20) & 15u) - 8), hi.z, s);
            s = fmaf((float)((int)(x >> 28) - 8), hi.w, s);
        }
        return s;
    }
};
// rows [r0, ...) of a [rows, K] weight matrix of type WT: K elements per row,
// or K / 2 bytes of Q4_0 codes
template <typename WT>
__device__ __forceinline__ const WT* weight_rows(const WT* W, long long r0, int K) {
    return W + r0 * K;
}
template <>
__device__ __forceinline__ const Q4Code* weight_rows<Q4Code>(const Q4Code* W, long long r0, int K) {
    return W + r0 * (K / 2);
}
// scale of chunk c of row r of a [rows, K] weight matrix: 1 unless quantised
template <typename WT>
__device__ __forceinline__ float chunk_scale(const uint16_t* S, long long r, int K, int c) {
    if constexpr (Chunk<WT>::QUANT) {
        return __half2float(__ushort_as_half(__ldg(S + r * (K / 32) + c / (32 / Chunk<WT>::EPC))));
    } else {
        return 1.f;
    }
}

// ---------------------------------------------------------------------------
// GEMV over a row range: out[r, b] = sum_c W[r, c] act[b, c] for b in
// [b0, b0 + NB) (masked by nb), one warp per row, grid-strided over rows.
// TWO = true also computes the same row of a second matrix W2 (GeGLU gate/up).
// ---------------------------------------------------------------------------
template <typename WT, int U, int NB, bool TWO, class Epi>
__device__ __forceinline__ void gemv_rows(const WT* __restrict__ W, const WT* __restrict__ W2, int rows, int K,
                                          const float* act, int lda, int b0, int nb, Epi& epi,
                                          const uint16_t* S = nullptr, const uint16_t* S2 = nullptr) {
    constexpr int EPC = Chunk<WT>::EPC;
    const int nch = K / EPC;
    const int lane = threadIdx.x & 31;
    const int gw = blockIdx.x * kWarps + (threadIdx.x >> 5);
    const int nw = gridDim.x * kWarps;
    const unsigned long long pol = l2_evict_first();
    for (int r = gw; r < rows; r += nw) {
        const uint4* wr = reinterpret_cast<const uint4*>(weight_rows(W, r, K));
        const uint4* wr2 = TWO ? reinterpret_cast<const uint4*>(weight_rows(W2, r, K)) : nullptr;
        float acc[NB], acc2[NB];
#pragma unroll
        for (int j = 0; j < NB; ++j) { acc[j] = 0.f; acc2[j] = 0.f; }
        for (int c0 = 0; c0 < nch; c0 += 32 * U) {
            uint4 w[U], w2[TWO ? U : 1];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + lane + 32 * u;
                w[u] = c < nch ? ld_weight16(wr + c, pol) : make_uint4(0u, 0u, 0u, 0u);
                if (TWO) w2[u] = c < nch ? ld_weight16(wr2 + c, pol) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + lane + 32 * u;
                if (c < nch) {
                    const float sc = chunk_scale<WT>(S, r, K, c);
                    const float sc2 = TWO ? chunk_scale<WT>(S2, r, K, c) : 1.f;
#pragma unroll
                    for (int j = 0; j < NB; ++j) {
                        if (b0 + j < nb) {
                            const float* a = act + (long long)(b0 + j) * lda + c * EPC;
                            acc[j] += Chunk<WT>::dot(w[u], a) * sc;
                            if (TWO) acc2[j] += Chunk<WT>::dot(w2[u], a) * sc2;
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

// One sequence, fewer rows than half the grid's warps: S warps of a CTA
// share a row, each over a contiguous 1/S of its chunks, and the partial dot
// products are added in segment order through `xred` (kWarps floats).
template <typename WT, int U, int S, class Epi>
__device__ __forceinline__ void gemv_rows_split(const WT* __restrict__ W, int rows, int K, const float* act, Epi& epi,
                                                float* xred, const uint16_t* SW = nullptr) {
    constexpr int EPC = Chunk<WT>::EPC, RPC = kWarps / S;
    const int nch = K / EPC;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, seg = warp % S;
    const int c_lo = seg * nch / S, c_hi = (seg + 1) * nch / S;
    const unsigned long long pol = l2_evict_first();
    for (int r0 = blockIdx.x * RPC; r0 < rows; r0 += gridDim.x * RPC) {   // the same trip count on every warp
        const int r = r0 + warp / S;
        float acc = 0.f;
        if (r < rows) {
            const uint4* wr = reinterpret_cast<const uint4*>(weight_rows(W, r, K));
            for (int c0 = c_lo; c0 < c_hi; c0 += 32 * U) {
                uint4 w[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int c = c0 + lane + 32 * u;
                    w[u] = c < c_hi ? ld_weight16(wr + c, pol) : make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int c = c0 + lane + 32 * u;
                    if (c < c_hi) acc += Chunk<WT>::dot(w[u], act + c * EPC) * chunk_scale<WT>(SW, r, K, c);
                }
            }
            acc = warp_sum(acc);
        }
        if (seg != 0 && lane == 0) xred[warp] = acc;
        __syncthreads();
        if (seg == 0 && r < rows) {
#pragma unroll
            for (int q = 1; q < S; ++q) acc += xred[warp + q];
            const float a[1] = {acc};
            epi.apply(r, 0, 1, a, a);
        }
        __syncthreads();
    }
}

// One sequence, rows of at most 16 U chunks: each warp loads two of its
// grid-strided rows (r and r + the grid's warp count) in one batch.
template <typename WT, int U, class Epi>
__device__ __forceinline__ void gemv_rows_pair(const WT* __restrict__ W, int rows, int K, const float* act, Epi& epi,
                                               const uint16_t* SW = nullptr) {
    constexpr int EPC = Chunk<WT>::EPC, UH = U / 2;
    const int nch = K / EPC;
    const int lane = threadIdx.x & 31;
    const int gw = blockIdx.x * kWarps + (threadIdx.x >> 5);
    const int nw = gridDim.x * kWarps;
    const unsigned long long pol = l2_evict_first();
    for (int r = gw; r < rows; r += 2 * nw) {
        const int r2 = r + nw;
        const bool two = r2 < rows;
        const uint4* wa = reinterpret_cast<const uint4*>(weight_rows(W, r, K));
        const uint4* wb = reinterpret_cast<const uint4*>(weight_rows(W, two ? r2 : r, K));
        uint4 w[U];
#pragma unroll
        for (int u = 0; u < UH; ++u) {
            const int c = lane + 32 * u;
            w[u] = c < nch ? ld_weight16(wa + c, pol) : make_uint4(0u, 0u, 0u, 0u);
            w[UH + u] = c < nch && two ? ld_weight16(wb + c, pol) : make_uint4(0u, 0u, 0u, 0u);
        }
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int u = 0; u < UH; ++u) {
            const int c = lane + 32 * u;
            if (c < nch) {
                a0 += Chunk<WT>::dot(w[u], act + c * EPC) * chunk_scale<WT>(SW, r, K, c);
                a1 += Chunk<WT>::dot(w[UH + u], act + c * EPC) * chunk_scale<WT>(SW, two ? r2 : r, K, c);
            }
        }
        const float s0[1] = {warp_sum(a0)}, s1[1] = {warp_sum(a1)};
        epi.apply(r, 0, 1, s0, s0);
        if (two) epi.apply(r2, 0, 1, s1, s1);
    }
}

// S, S2: the block scales of W, W2 when WT is a quantised code type (Chunk::QUANT)
template <typename WT, int U, bool TWO, class Epi>
__device__ __forceinline__ void gemv(const WT* W, const WT* W2, int rows, int K, const float* act, int lda, int nb,
                                     Epi& epi, float* xred, const uint16_t* S = nullptr, const uint16_t* S2 = nullptr) {
    if (nb == 1) {
        const int nw = gridDim.x * kWarps, nch = K / Chunk<WT>::EPC;
        if (!TWO && 2 * rows <= nw && nch >= 64)
            gemv_rows_split<WT, U, 2>(W, rows, K, act, epi, xred, S);
        else if (!TWO && rows > nw && 2 * nch <= 32 * U)
            gemv_rows_pair<WT, U>(W, rows, K, act, epi, S);
        else
            gemv_rows<WT, U, 1, TWO>(W, W2, rows, K, act, lda, 0, 1, epi, S, S2);
    } else {
        for (int b0 = 0; b0 < nb; b0 += 4) gemv_rows<WT, U, 4, TWO>(W, W2, rows, K, act, lda, b0, nb, epi, S, S2);
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

// Tensor-core operand rows (batch b, column k) live in global memory in the
// shared-memory image of the MMA's K-major 128-byte-swizzled tiles: per K
// block of 64 columns, Bp rows of 128 bytes with 16-byte chunk c of row b
// at chunk position c ^ (b % 8), so one bulk copy of a block lands ready
// for the MMA.  Element index of (b, k):
__device__ __forceinline__ long long xtile_idx(int b, int k, int Bp) {
    const int kb = k >> 6, kk = k & 63;
    return ((long long)kb * Bp + b) * 64 + ((((kk >> 3) ^ (b & 7)) << 3) | (kk & 7));
}

// out[b * ldo + r] = v, plus the bf16 high and low parts of v as
// tensor-core operand elements (b, r)
struct StoreXhEpi {
    float* out;
    int ldo;
    uint16_t *xh, *xl;
    int Bp;
    template <int NB>
    __device__ __forceinline__ void apply(int r, int b0, int nb, const float (&acc)[NB], const float (&)[NB]) {
        const int lane = threadIdx.x & 31;
#pragma unroll
        for (int j = 0; j < NB; ++j)
            if (lane == j && b0 + j < nb) {
                const float v = acc[j];
                out[(long long)(b0 + j) * ldo + r] = v;
                const long long xi = xtile_idx(b0 + j, r, Bp);
                const __nv_bfloat16 hi = __float2bfloat16_rn(v);
                xh[xi] = __bfloat16_as_ushort(hi);
                xl[xi] = __bfloat16_as_ushort(__float2bfloat16_rn(v - __bfloat162float(hi)));
            }
    }
};

__device__ __forceinline__ float gelu_tanh(float x) {
    const float k0 = 0.7978845608028654f;  // sqrt(2 / pi)
    return 0.5f * x * (1.f + tanhf(k0 * (x + 0.044715f * x * x * x)));
}

__device__ __forceinline__ float silu(float x) { return x / (1.f + expf(-x)); }

// m[b * ldo + r] = gelu_tanh(gate) * up, or (NextN) silu(gate) * up
struct GegluEpi {
    float* out;
    int ldo;
    int swiglu;
    template <int NB>
    __device__ __forceinline__ void apply(int r, int b0, int nb, const float (&g)[NB], const float (&u)[NB]) {
        const int lane = threadIdx.x & 31;
#pragma unroll
        for (int j = 0; j < NB; ++j)
            if (lane == j && b0 + j < nb)
                out[(long long)(b0 + j) * ldo + r] = (swiglu ? silu(g[j]) : gelu_tanh(g[j])) * u[j];
    }
};

// Running softmax denominator of a stream of logits: m the largest seen, s
// the sum of exp(z - m) (NaN left out).  Two partials merge exactly.
struct SoftDen {
    float m, s;
    __device__ __forceinline__ void add(float z) {
        if (!(z == z)) return;
        if (z > m) {
            s = s * expf(m - z) + 1.f;   // m = -inf: s = 0 * 0 + 1
            m = z;
        } else {
            s += expf(z - m);
        }
    }
    __device__ __forceinline__ void merge(float m2, float s2) {
        if (!(s2 > 0.f)) return;
        if (!(s > 0.f)) {
            m = m2;
            s = s2;
        } else if (m2 > m) {
            s = s * expf(m - m2) + s2;
            m = m2;
        } else {
            s += s2 * expf(m2 - m);
        }
    }
};
__device__ __forceinline__ SoftDen soft_den0() { return SoftDen{-INFINITY, 0.f}; }

// LM head: softcap, optional logits store, running packed argmax per column
// (lane c & 31 owns column c; two registers cover 64 columns), and with
// `conf` the columns' running softmax denominators.
struct HeadEpi {
    float* logits;  // [B, N, V] or null
    int V, N, step;
    float softcap;
    unsigned long long best_lo, best_hi;
    float* zb;      // [B, V] the step's logits for the sampler, or null
    bool conf;      // keep the softmax denominators (per-step confidence output)
    SoftDen den_lo, den_hi;
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
                if (zb) zb[(long long)col * V + r] = z;
                const unsigned long long k = pack_argmax(z, (uint32_t)r);
                if (col < 32) best_lo = k > best_lo ? k : best_lo;
                else best_hi = k > best_hi ? k : best_hi;
                if (conf) {
                    if (col < 32) den_lo.add(z);
                    else den_hi.add(z);
                }
            }
        }
    }
};

// ---------------------------------------------------------------------------
// prologues: build one sequence's GEMV input vector
// ---------------------------------------------------------------------------

// dst[i] = src[i] * rsqrt(mean(src^2) + eps) * gs[i] with the gains staged in
// shared memory (gs); src may alias dst.  All threads of the CTA participate.
__device__ __forceinline__ void rms_into_s(const float* src, const float* gs, int n, float eps, float* dst, float* red) {
    float ss = 0.f;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const float v = src[i];
        ss = fmaf(v, v, ss);
    }
    ss = block_sum(ss, red);
    const float r = 1.0f / sqrtf(ss / (float)n + eps);
    for (int i = threadIdx.x; i < n; i += blockDim.x) dst[i] = src[i] * r * gs[i];
    __syncthreads();
}

// Both halves of v[2n] RMS-normalised in place with staged gains gs[2n]
// (one block reduction for the two sums; red holds 2 kWarps floats).
__device__ __forceinline__ void rms_pair_s(float* v, const float* gs, int n, float eps, float* red) {
    float s1 = 0.f, s2 = 0.f;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const float a = v[i], c = v[n + i];
        s1 = fmaf(a, a, s1);
        s2 = fmaf(c, c, s2);
    }
    s1 = warp_sum(s1);
    s2 = warp_sum(s2);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    __syncthreads();
    if (lane == 0) {
        red[warp] = s1;
        red[kWarps + warp] = s2;
    }
    __syncthreads();
    s1 = warp_sum(lane < kWarps ? red[lane] : 0.f);
    s2 = warp_sum(lane < kWarps ? red[kWarps + lane] : 0.f);
    const float r1 = 1.0f / sqrtf(s1 / (float)n + eps), r2 = 1.0f / sqrtf(s2 / (float)n + eps);
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        v[i] = v[i] * r1 * gs[i];
        v[n + i] = v[n + i] * r2 * gs[n + i];
    }
    __syncthreads();
}

// token consumed by sequence b at step k
__device__ __forceinline__ int step_token(const DraftParams& p, int b, int k) {
    if (k == 0) return p.last_tok[b];
    const uint32_t t = unpack_index(__ldcg(p.amax + (long long)(k - 1) * p.B + b));
    return t < (uint32_t)p.V ? (int)t : 0;   // every slot holds a row index after its HEAD phase
}

// NextN: the catch-up row of sequence b at iteration k < 0 (rows are
// right-aligned: iteration -1 takes the last), negative if b has none there
__device__ __forceinline__ int catchup_row(const DraftParams& p, int b, int k) {
    return (p.n_cu ? __ldg(p.n_cu + b) : 0) + k;
}
// Position of sequence b's row at iteration k: the query position
// kv_len + k of the assistant's draft steps; for NextN the row index in its
// own KV, kv_len + j for catch-up row j, kv_len + n_cu + k for draft step k
__device__ __forceinline__ int row_pos(const DraftParams& p, const int* kv, int b, int k) {
    if (!p.nextn) return kv[b] + k;
    const int j = catchup_row(p, b, k);
    return kv[b] + (j > 0 ? j : 0);
}

// float4 at q summed over S copies st floats apart, in order
__device__ __forceinline__ float4 ld4_sum(const float* q, int S, long long st) {
    float4 a = __ldcg(reinterpret_cast<const float4*>(q));
    int s = 1;
    for (; s + 4 <= S; s += 4) {   // four loads in flight, summed in order
        float4 c[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) c[u] = __ldcg(reinterpret_cast<const float4*>(q + (s + u) * st));
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            a.x += c[u].x;
            a.y += c[u].y;
            a.z += c[u].z;
            a.w += c[u].w;
        }
    }
    for (; s < S; ++s) {
        const float4 c = __ldcg(reinterpret_cast<const float4*>(q + s * st));
        a.x += c.x;
        a.y += c.y;
        a.z += c.z;
        a.w += c.w;
    }
    return a;
}

// dst[i] = sum over s < S of sequence b's split partial i (tensor-core
// projection with R output rows), i < n, n a multiple of 4.  The CTA's
// threads take float4 columns; when there are fewer columns than threads,
// each column's partials are cut into G contiguous groups summed in order by
// G threads (up to 8 loads in flight each), and the group sums are added in
// group order through scratch[G n] -- a fixed order, so the result is
// deterministic.  Synchronises the CTA.
static __device__ __noinline__ void part_sum_vec(const DraftParams& p, int S, int R, int b, int n, float* dst,
                                             float* scratch) {
    const int ncol = n >> 2;
    int G = (int)blockDim.x / (ncol > 0 ? ncol : 1);
    G = G < 1 ? 1 : (G > 4 ? 4 : G);
    const int per = (S + G - 1) / G;
    const long long st = (long long)p.B * R;
    const float* base = p.PB + (long long)b * R;
    for (int t = threadIdx.x; t < ncol * G; t += blockDim.x) {
        const int c = t % ncol, g = t / ncol;
        const int s0 = g * per, s1 = s0 + per < S ? s0 + per : S;
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int sb = s0; sb < s1; sb += 8) {
            float4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (sb + u < s1) v[u] = __ldcg(reinterpret_cast<const float4*>(base + (sb + u) * st) + c);
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (sb + u < s1) {
                    a.x += v[u].x;
                    a.y += v[u].y;
                    a.z += v[u].z;
                    a.w += v[u].w;
                }
        }
        reinterpret_cast<float4*>(G == 1 ? dst : scratch + (long long)g * n)[c] = a;
    }
    __syncthreads();
    if (G > 1) {
        for (int c = threadIdx.x; c < ncol; c += blockDim.x) {
            float4 a = reinterpret_cast<const float4*>(scratch)[c];
            for (int g = 1; g < G; ++g) {
                const float4 v = reinterpret_cast<const float4*>(scratch + (long long)g * n)[c];
                a.x += v.x;
                a.y += v.y;
                a.z += v.z;
                a.w += v.w;
            }
            reinterpret_cast<float4*>(dst)[c] = a;
        }
        __syncthreads();
    }
}

// dst[s][i] = src[s][i] for i < n (n a multiple of 4, 16-byte aligned rows):
// every load of a thread is issued before its first store.  The stores go
// through generic pointers the compiler cannot tell apart from the sources,
// so a loop that stored each element before loading the next would wait for
// one round trip per element.
template <int NS>
struct VecCopy {
    const float* src[NS];
    float* dst[NS];
};
// (global-memory sources only)
template <int NS, int MAXV>
__device__ __forceinline__ void vec_copy(const VecCopy<NS>& c, int n) {
    const int n4 = n >> 2;
#pragma unroll 1
    for (int base = threadIdx.x; base < n4; base += MAXV * kThreads) {
        float4 v[NS][MAXV];
#pragma unroll
        for (int j = 0; j < MAXV; ++j) {
            const int i = base + j * kThreads;
#pragma unroll
            for (int s = 0; s < NS; ++s)
                if (i < n4) v[s][j] = __ldcg(reinterpret_cast<const float4*>(c.src[s]) + i);
        }
#pragma unroll
        for (int j = 0; j < MAXV; ++j) {
            const int i = base + j * kThreads;
#pragma unroll
            for (int s = 0; s < NS; ++s)
                if (i < n4) reinterpret_cast<float4*>(c.dst[s])[i] = v[s][j];
        }
    }
}

// Writes sequence b's input vector for `phase` into dst (length phase_k).
// `writer` marks the one CTA that also stores residual-stream updates.  The
// norm gains are staged in gs (2 max(d_t, d_a) floats) by the same loops that
// load the activations.
struct AttnTab;
static __device__ void attn_fold_row(const DraftParams& p, const AttnTab& tab, int l, int b, float* dst);

template <typename WT, bool TC>
__device__ void build_act(const DraftParams& p, int phase, int k, int l, int b, float* dst, float* tmp, bool writer,
                          float* red, float* gs, const AttnTab* tab) {
    switch (phase) {
    case PH_PRE: {
        const int n = p.d_t;
        constexpr int EPC = 16 / (int)sizeof(WT);
        int tok;
        const float* h;
        if (k < 0) {
            // NextN catch-up iteration k: row n_cu + k of sequence b, or (none
            // at this iteration) the first step's inputs, computed and unused
            const int j = catchup_row(p, b, k);
            tok = j >= 0 ? __ldg(p.cu_tok + (long long)b * p.M + j) : p.last_tok[b];
            h = j >= 0 ? p.cu_h + ((long long)b * p.M + j) * n : p.h_prev + (long long)b * n;
        } else {
            tok = step_token(p, b, k);
            h = k == 0 ? p.h_prev + (long long)b * n : (p.nextn ? p.HX : p.HN) + (long long)b * n;
        }
        const uint4* er = reinterpret_cast<const uint4*>(reinterpret_cast<const WT*>(p.tok_embd) + (long long)tok * n);
#pragma unroll 2
        for (int j = threadIdx.x; j < n / EPC; j += blockDim.x) {   // the embedding row, 16-byte vectors
            const uint4 w = ld_stream16(er + j);
#pragma unroll
            for (int e = 0; e < EPC; ++e) dst[j * EPC + e] = Chunk<WT>::elem(w, e) * p.emb_scale;
        }
#pragma unroll 4
        for (int i = threadIdx.x; i < n; i += blockDim.x) {
            dst[n + i] = __ldcg(h + i);
            gs[i] = __ldg(p.norm_e + i);
            gs[n + i] = __ldg(p.norm_h + i);
        }
        __syncthreads();
        rms_pair_s(dst, gs, n, p.eps, red);
        break;
    }
    case PH_Q: {
        const int n = p.d_a;
        const float* ga = p.blk[l].attn_norm;
        if (l == 0) {
            if ((TC && p.tc_proj)) {   // the pre-projection's partials form the residual stream
                part_sum_vec(p, p.sk[PH_PRE], n, b, n, tmp, dst);
                for (int i = threadIdx.x; i < n; i += blockDim.x) {
                    gs[i] = __ldg(ga + i);
                    if (writer) p.XB[(long long)b * n + i] = tmp[i];
                }
            } else {
#pragma unroll 4
                for (int i = threadIdx.x; i < n; i += blockDim.x) {
                    tmp[i] = __ldcg(p.XB + (long long)b * n + i);
                    gs[i] = __ldg(ga + i);
                }
            }
            __syncthreads();
        } else {
            const float* gp = p.blk[l - 1].post_ffn_norm;
            if ((TC && p.tc_proj)) part_sum_vec(p, p.sk[PH_FFN2], n, b, n, dst, dst + n);
#pragma unroll 4
            for (int i = threadIdx.x; i < n; i += blockDim.x) {
                if (!(TC && p.tc_proj)) dst[i] = __ldcg(p.Y2 + (long long)b * n + i);
                tmp[i] = __ldcg(p.XM + (long long)b * n + i);
                gs[i] = __ldg(ga + i);
                gs[n + i] = __ldg(gp + i);
            }
            __syncthreads();
            rms_into_s(dst, gs + n, n, p.eps, dst, red);
            for (int i = threadIdx.x; i < n; i += blockDim.x) {
                const float x = tmp[i] + dst[i];
                tmp[i] = x;
                if (writer) p.XB[(long long)b * n + i] = x;
            }
            __syncthreads();
        }
        rms_into_s(tmp, gs, n, p.eps, dst, red);
        break;
    }
    case PH_FFN1: {
        const int n = p.d_a;
        const float *g1 = p.blk[l].post_attn_norm, *g2 = p.blk[l].pre_ffn_norm;
        if ((TC && p.tc_proj)) part_sum_vec(p, p.sk[PH_O], n, b, n, dst, dst + n);
#pragma unroll 4
        for (int i = threadIdx.x; i < n; i += blockDim.x) {
            if (!(TC && p.tc_proj)) dst[i] = __ldcg(p.YB + (long long)b * n + i);
            tmp[i] = __ldcg(p.XB + (long long)b * n + i);
            if (!p.nextn) gs[i] = __ldg(g1 + i);
            gs[n + i] = __ldg(g2 + i);
        }
        __syncthreads();
        if (!p.nextn) rms_into_s(dst, gs, n, p.eps, dst, red);   // NextN: the attention output added as it is
        for (int i = threadIdx.x; i < n; i += blockDim.x) {
            const float x = tmp[i] + dst[i];
            tmp[i] = x;
            if (writer) p.XM[(long long)b * n + i] = x;
        }
        __syncthreads();
        rms_into_s(tmp, gs + n, n, p.eps, dst, red);
        break;
    }
    case PH_POST: {
        const int n = p.d_a;
        const float *g1 = p.blk[p.L - 1].post_ffn_norm, *g2 = p.final_norm;
        if ((TC && p.tc_proj)) part_sum_vec(p, p.sk[PH_FFN2], n, b, n, dst, dst + n);
#pragma unroll 4
        for (int i = threadIdx.x; i < n; i += blockDim.x) {
            if (!(TC && p.tc_proj)) dst[i] = __ldcg(p.Y2 + (long long)b * n + i);
            tmp[i] = __ldcg(p.XM + (long long)b * n + i);
            gs[i] = __ldg(g1 + i);
            gs[n + i] = __ldg(g2 + i);
        }
        __syncthreads();
        rms_into_s(dst, gs, n, p.eps, dst, red);
        for (int i = threadIdx.x; i < n; i += blockDim.x) tmp[i] += dst[i];
        __syncthreads();
        rms_into_s(tmp, gs + n, n, p.eps, dst, red);
        break;
    }
    case PH_O: {
        const int n = p.Hq * p.hd;
        if (p.att_fold) attn_fold_row(p, *tab, l, b, dst);   // merges the attention's split partials here
        else vec_copy<1, 1>(VecCopy<1>{{p.OB + (long long)b * n}, {dst}}, n);
        __syncthreads();
        break;
    }
    case PH_FFN2: {
        const int n = p.F;
        if ((TC && p.tc_proj)) {   // GeGLU of the summed gate (rows 0..F-1) and up (rows F..2F-1) partials
            const long long st = (long long)p.B * 2 * n;
            const float* q = p.PB + (long long)b * 2 * n;
            const int S = p.sk[PH_FFN1];
            for (int i4 = threadIdx.x; i4 < (n >> 2); i4 += kThreads) {
                const float4 g = ld4_sum(q + 4 * i4, S, st), u = ld4_sum(q + n + 4 * i4, S, st);
                if (p.nextn)
                    reinterpret_cast<float4*>(dst)[i4] = make_float4(silu(g.x) * u.x, silu(g.y) * u.y, silu(g.z) * u.z,
                                                                     silu(g.w) * u.w);
                else
                    reinterpret_cast<float4*>(dst)[i4] = make_float4(gelu_tanh(g.x) * u.x, gelu_tanh(g.y) * u.y,
                                                                     gelu_tanh(g.z) * u.z, gelu_tanh(g.w) * u.w);
            }
        } else {
            vec_copy<1, 1>(VecCopy<1>{{p.MB + (long long)b * n}, {dst}}, n);
        }
        __syncthreads();
        break;
    }
    case PH_HEAD: {
        const int n = p.d_t;
        vec_copy<1, 1>(VecCopy<1>{{p.HN + (long long)b * n}, {dst}}, n);
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
template <typename WT, bool TC>
__device__ const float* stage_act(const DraftParams& p, int phase, int k, int l, float* smem_act, float* smem_tmp,
                                  float* red, unsigned int& epoch, int& lda, bool& ok, const AttnTab* tab) {
    const int K = phase_k(p, phase);
    // gain stage after the activation area
    float* gs = smem_act + (p.act_smem ? (long long)p.B * p.kmax : (long long)p.kmax);
    ok = true;
    if (p.act_smem) {
        for (int b = 0; b < p.B; ++b)
            build_act<WT, TC>(p, phase, k, l, b, smem_act + (long long)b * K, smem_tmp, blockIdx.x == 0, red, gs, tab);
        lda = K;
        return smem_act;
    }
    // global mode: copy-only inputs are read in place
    if (!(TC && p.tc_proj)) {
        if (phase == PH_O) { lda = K; return p.OB; }
        if (phase == PH_FFN2) { lda = K; return p.MB; }
        if (phase == PH_HEAD) { lda = K; return p.HN; }
    }
    for (int b = blockIdx.x; b < p.B; b += gridDim.x) {
        build_act<WT, TC>(p, phase, k, l, b, smem_act, smem_tmp, true, red, gs, tab);
        if ((TC && p.tc_proj)) {
            // tensor-core operand: bf16 high and low parts, read by tensor
            // copies; 8 consecutive columns are one 16-byte chunk of the
            // swizzled tile, stored at once (K is a multiple of 8)
            for (int c = threadIdx.x; c < K / 8; c += blockDim.x) {
                const float4 v0 = reinterpret_cast<const float4*>(smem_act)[2 * c];
                const float4 v1 = reinterpret_cast<const float4*>(smem_act)[2 * c + 1];
                const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
                uint32_t hw[4], lw[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const __nv_bfloat16 h0 = __float2bfloat16_rn(v[2 * e]), h1 = __float2bfloat16_rn(v[2 * e + 1]);
                    const __nv_bfloat16 l0 = __float2bfloat16_rn(v[2 * e] - __bfloat162float(h0));
                    const __nv_bfloat16 l1 = __float2bfloat16_rn(v[2 * e + 1] - __bfloat162float(h1));
                    hw[e] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
                    lw[e] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
                }
                const long long xi = xtile_idx(b, 8 * c, p.Bp);
                *reinterpret_cast<uint4*>(p.XA + xi) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                *reinterpret_cast<uint4*>(p.XAL + xi) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
            }
            fence_proxy_async_global();
        } else {
            for (int i = threadIdx.x; i < K; i += blockDim.x) p.ACT[(long long)b * p.kmax + i] = smem_act[i];
        }
        __syncthreads();
    }
    ok = grid_barrier(p.hdr, epoch, p.timeout_ns, gridDim.x);
    lda = p.kmax;
    return p.ACT;
}

// first row of CTA c's block of R rows
__device__ __forceinline__ int row_lo(int R, int c) { return (int)(((long long)R * c) / gridDim.x); }

// Bounded wait on an mbarrier phase: false once limit_ns passed.
__device__ __forceinline__ bool mbar_wait_limited(unsigned long long* bar, unsigned int parity,
                                                  unsigned long long limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_ns() - t0 > limit_ns) return false;
    return true;
}

// ---------------------------------------------------------------------------
// attention: flash decoding, split over key ranges
// ---------------------------------------------------------------------------
// An item is (sequence b, KV head g, key range).  The CTA's warps take R-key
// slices of the range round-robin; every warp streams its slices through a
// private two-stage cp.async ring in shared memory and keeps its own
// online-softmax state (m, l, o) for HG query heads of the group at a time,
// with the lanes of one K/V row splitting the head dimension.  The warps are
// merged in shared memory.  An (b, g) with one item writes OB directly;
// otherwise every item stores its (o, m, l) in PART and counts itself in
// att_cnt[b, g], and once the CTA has stored all its items it waits for the
// count of each of them and merges the item's share of the outputs.  No CTA
// waits before all its own items are stored, so the waits always end.

__device__ __forceinline__ int view_lo(const KView& v, int kv_len) {
    return (v.window > 0 && kv_len > v.window) ? kv_len - v.window : 0;
}

// A sequence's keys in a view ("opus-mtp-turbo: Track 1 report", item 2,
// sink + window): key index x < s0 is position x (the attention sink,
// positions [0, min(sink, lo))), key index x >= s0 is position lo + x - s0
// (the window [lo, kv_len)).  Position t lives in slot t below the sink and
// in slot sink + (t - sink) % (cap - sink) from it on (a plain ring when
// sink = 0).
struct KeyMap {
    int lo, s0, sink, cap, n;   // window start, sink keys, sink, slots, keys
    unsigned int ring, magic;   // cap - sink and floor(2^32 / ring): d % ring by a multiply-high
};
__device__ __forceinline__ KeyMap key_map(const KView& v, int kv_len) {
    KeyMap m;
    m.lo = view_lo(v, kv_len);
    m.s0 = v.window > 0 ? (v.sink < m.lo ? v.sink : m.lo) : 0;
    m.sink = v.window > 0 ? v.sink : 0;
    m.cap = v.cap;
    m.n = m.s0 + kv_len - m.lo;
    m.ring = (unsigned int)(m.cap - m.sink);
    m.magic = v.window > 0 ? v.ring_magic : v.cap_magic;
    return m;
}
__device__ __forceinline__ int view_keys(const KView& v, int kv_len) { return key_map(v, kv_len).n; }
// d % ring for 0 <= d < 2^31: the multiply-high quotient is exact or one short
__device__ __forceinline__ unsigned int ring_mod(const KeyMap& m, unsigned int d) {
    unsigned int r = d - __umulhi(d, m.magic) * m.ring;
    return r >= m.ring ? r - m.ring : r;
}
__device__ __forceinline__ int key_slot(const KeyMap& m, int x) {
    const int t = x < m.s0 ? x : m.lo + (x - m.s0);
    return t < m.sink ? t : m.sink + (int)ring_mod(m, (unsigned int)(t - m.sink));
}
// keys from x on (at most `limit`) whose slots follow one another; `slot` is key x's slot
__device__ __forceinline__ int key_run(const KeyMap& m, int x, int slot, int limit) {
    int run = limit;
    if (x < m.s0 && m.s0 - x < run) run = m.s0 - x;   // the sink keys end
    const int rs = m.cap - slot;                      // the ring wraps
    return rs < run ? rs : run;
}

// Key-space partition of an attention phase, per view (the sequence lengths
// are fixed for a launch): the (sequence b, KV head g) segments lie end to
// end in b-major order, segment (b, g) holding sequence b's n_b readable
// keys, T keys in all; CTA c < G takes positions [T c / G, T (c + 1) / G).
// G is the grid, or fewer CTAs where that would leave each under 16 R keys.
// A piece is the part of one segment inside one CTA's range.
// When every segment has the same length and there are no more segments
// than CTAs, each segment instead gets cseg CTAs of its own (one piece each).
struct AttnTab {
    long long T[MTP_MAX_VIEWS];
    int G[MTP_MAX_VIEWS], cseg[MTP_MAX_VIEWS];
    long long pre[MTP_MAX_VIEWS][MTP_MAX_BATCH + 1];   // positions before sequence b's segments
};
// thread v < MTP_MAX_VIEWS fills view v (R: keys per warp slice)
__device__ __forceinline__ void attn_tab_fill(const DraftParams& p, const int* kv, int R, AttnTab& t) {
    const int v = threadIdx.x;
    if (v >= MTP_MAX_VIEWS) return;
    const KView& vw = p.views[v];
    long long T = 0;
    for (int b = 0; b < p.B; ++b) {
        t.pre[v][b] = T;
        T += (long long)view_keys(vw, kv[b]) * p.Hkv;
    }
    t.pre[v][p.B] = T;
    long long G = T / ((long long)kWarps * R);
    if (G > (long long)gridDim.x) G = gridDim.x;
    if (G < 1) G = 1;
    t.T[v] = T;
    t.G[v] = (int)G;
    // equal segments: whole CTAs per segment
    const int n0 = view_keys(vw, kv[0]), nseg = p.B * p.Hkv;
    bool equal = true;
    for (int b = 1; b < p.B; ++b) equal = equal && view_keys(vw, kv[b]) == n0;
    int c = nseg <= (int)gridDim.x ? (int)gridDim.x / nseg : 0;
    if (c > n0 / (kWarps * R)) c = n0 / (kWarps * R);
    t.cseg[v] = equal && c >= 1 ? c : 0;
}
// first position of CTA c's range, and the CTA whose range holds position x
__device__ __forceinline__ long long attn_lo(const AttnTab& t, int v, int c) { return t.T[v] * c / t.G[v]; }
__device__ __forceinline__ int attn_cta(const AttnTab& t, int v, long long x) {
    return (int)(((x + 1) * t.G[v] - 1) / t.T[v]);
}

struct AttnPiece {
    int b, g, t_beg, t_end;   // key indices [t_beg, t_end) of KV head g of sequence b (see KeyMap)
    int cf, S;                // first CTA over the segment and their count (S == 1: one piece)
    int slot;                 // partial slot of this piece: 2 c, or 2 c + 1 for a range's last piece
};
// CTA c's piece starting at position x; `next` = position after it
__device__ __forceinline__ AttnPiece attn_piece(const DraftParams& p, const KView& vw, const int* kv,
                                                const AttnTab& t, int v, int c, long long x, long long& next) {
    // the sequence holding x: the last b with pre[b] <= x (binary search)
    int b = 0;
    for (int hi = p.B - 1; b < hi;) {
        const int mid = (b + hi + 1) >> 1;
        if (t.pre[v][mid] <= x) b = mid;
        else hi = mid - 1;
    }
    const int n = view_keys(vw, kv[b]);
    const int g = (int)((x - t.pre[v][b]) / n);
    const long long s0 = t.pre[v][b] + (long long)g * n, s1 = s0 + n;
    const long long ce = attn_lo(t, v, c + 1);
    next = s1 < ce ? s1 : ce;
    AttnPiece P;
    P.b = b;
    P.g = g;
    P.t_beg = (int)(x - s0);
    P.t_end = (int)(next - s0);
    P.cf = attn_cta(t, v, s0);
    P.S = attn_cta(t, v, s1 - 1) - P.cf + 1;
    // a split segment is the first piece of every CTA over it but the
    // first one, whose range began in an earlier segment unless it starts
    // exactly at the segment
    P.slot = 2 * c + ((c == P.cf && attn_lo(t, v, c) != s0) ? 1 : 0);
    return P;
}
// equal segments: the piece of CTA c (c < B Hkv cseg)
__device__ __forceinline__ AttnPiece attn_piece_eq(const DraftParams& p, const KView& vw, const int* kv,
                                                   const AttnTab& t, int v, int c) {
    const int cs = t.cseg[v], j = c / cs, sp = c - j * cs;
    AttnPiece P;
    P.b = j / p.Hkv;
    P.g = j - P.b * p.Hkv;
    // even split: the first n % cs pieces take one key more
    const int n = view_keys(vw, kv[P.b]), q = n / cs, r = n - q * cs;
    P.t_beg = sp * q + (sp < r ? sp : r);
    P.t_end = P.t_beg + q + (sp < r ? 1 : 0);
    P.cf = j * cs;
    P.S = cs;
    P.slot = 2 * c;
    return P;
}
// partial slot of the q-th CTA over a split segment starting at position s0
__device__ __forceinline__ int attn_slot(const AttnTab& t, int v, int cf, int q, long long s0) {
    if (t.cseg[v] > 0) return 2 * (cf + q);
    return 2 * (cf + q) + ((q == 0 && attn_lo(t, v, cf) != s0) ? 1 : 0);
}

// The attention output of sequence b for block l, [Hq][hd], into dst (whole
// CTA): per (b, KV head g) segment the finished output when one CTA covered
// it, else the LSE merge of its CTAs' partials.  Used by the O prologue when
// the attention phase leaves its split segments unmerged (att_fold).  One
// warp per head: lanes take the partials' (m, l) in parallel, then the
// head's hd outputs (hd / 32 per lane) accumulate over the partials with
// every lane's loads of a partial in flight together.
static __device__ void attn_fold_row(const DraftParams& p, const AttnTab& tab, int l, int b, float* dst) {
    const int view = p.blk[l].view, HD = p.hd, grp = p.Hq / p.Hkv, PSZ = attn_psz(grp, HD);
    // keys per KV head of sequence b, as the attention's table counted them
    const int n = (int)((tab.pre[view][b + 1] - tab.pre[view][b]) / p.Hkv);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5, DL = HD / 32;
    for (int h = warp; h < p.Hq; h += nw) {
        const int g = h / grp, hh = h - g * grp;
        long long s0;
        int cf, S;
        if (tab.cseg[view] > 0) {
            const int cs = tab.cseg[view];
            cf = (b * p.Hkv + g) * cs;
            S = cs;
            s0 = 0;
        } else {
            s0 = tab.pre[view][b] + (long long)g * n;
            cf = attn_cta(tab, view, s0);
            S = attn_cta(tab, view, s0 + n - 1) - cf + 1;
        }
        float* out = dst + h * HD;
        if (S == 1) {
            for (int d = lane; d < HD; d += 32) out[d] = __ldcg(p.OB + ((long long)b * p.Hq + h) * HD + d);
            continue;
        }
        auto part = [&](int q) { return p.PART + (long long)attn_slot(tab, view, cf, q, s0) * PSZ; };
        float M = -INFINITY;
        for (int q = lane; q < S; q += 32) M = fmaxf(M, __ldcg(part(q) + grp * HD + hh));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        const float mu = M == -INFINITY ? 0.f : M;
        float Ls = 0.f, O[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) O[i] = 0.f;
        for (int q0 = 0; q0 < S; q0 += 32) {
            const int q = q0 + lane;
            float e = 0.f;
            if (q < S) {
                const float* pq = part(q);
                e = expf(__ldcg(pq + grp * HD + hh) - mu);
                Ls = fmaf(e, __ldcg(pq + grp * HD + grp + hh), Ls);
            }
            const int nq = S - q0 < 32 ? S - q0 : 32;
#pragma unroll 2
            for (int j = 0; j < nq; ++j) {
                const float ej = __shfl_sync(0xffffffffu, e, j);
                const float* oq = part(q0 + j) + hh * HD + lane;
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (i < DL) O[i] = fmaf(ej, __ldcg(oq + 32 * i), O[i]);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, o);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (i < DL) out[lane + 32 * i] = O[i] / Ls;
    }
}

// Sum of NV per-lane values over the LPR lanes of a row group, transposed:
// afterwards value idx = (lane % LPR) >> log2(LPR / NV) holds the group's
// total (high index bits from the high lane bits).  NV <= LPR, powers of 2.
template <int NV, int LPR>
__device__ __forceinline__ float transpose_sum(float (&v)[NV]) {
    static_assert(NV <= LPR, "transpose_sum needs NV <= LPR");
    const int lane = threadIdx.x & 31;
    float x[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) x[i] = v[i];
    int n = NV;
#pragma unroll
    for (int off = LPR / 2; off >= LPR / NV; off >>= 1) {
        n >>= 1;
        const bool up = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < NV / 2; ++i) {
            if (i < n) {
                const float send = up ? x[i] : x[i + n];
                const float keep = up ? x[i + n] : x[i];
                x[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
            }
        }
    }
    float r = x[0];
#pragma unroll
    for (int off = LPR / NV / 2; off >= 1; off >>= 1) r += __shfl_xor_sync(0xffffffffu, r, off);
    return r;
}

// Waits (thread 0) until *cnt reaches target; false when the time limit
// passed or another CTA reported an error.  Called by the whole CTA.
__device__ __forceinline__ bool count_wait(const unsigned int* cnt, unsigned int target, WsHeader* hdr,
                                           unsigned long long limit_ns) {
    __shared__ int s_ok;
    if (threadIdx.x == 0) {
        const unsigned long long t0 = global_ns();
        int ok = 1;
        unsigned int spins = 0;
        while (ld_acquire(cnt) < target) {
            if (ld_relaxed(&hdr->status) != 0) { ok = 0; break; }
            if ((++spins & 63u) == 0 && global_ns() - t0 > limit_ns) {
                atomicCAS(&hdr->status, 0, MTP_ERR_TIMEOUT);
                ok = 0;
                break;
            }
        }
        __threadfence();
        s_ok = ok;
    }
    __syncthreads();
    return s_ok != 0;
}

// release-add: the CTA's earlier writes (ordered by the preceding CTA
// barrier) become visible at GPU scope before the count
__device__ __forceinline__ void red_release_add(unsigned int* p, unsigned int v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// NST: ring stages per warp.  abar: [kWarps][NST] stage barriers (one arrival
// each); apar: the calling warp's stage phase bits, carried across calls.
template <typename WT, int HD, int NST>
__device__ __forceinline__ bool attention_body(const DraftParams& p, int l, unsigned char* smem, const int* kv, const AttnTab& tab,
                                unsigned long long* abar, unsigned int& apar) {
    constexpr AttnGeom G = attn_geom(HD, (int)sizeof(WT));
    constexpr int RB = G.RB, LPR = G.LPR, CPL = G.CPL, KPW = G.KPW, EPC = G.EPC, DPL = G.DPL;
    constexpr int R = G.R, RL = G.RL, SB = G.SB, HG = G.HG;
    constexpr int RING = kWarps * NST * SB;
    constexpr int NV = RL * HG;         // scores per lane and round
    // one K/V row per warp and NV <= 32: scores summed transposed, softmax on
    // one lane per score, probabilities broadcast through shared memory
    constexpr bool TR = KPW == 1 && NV <= LPR;
    constexpr int SH = TR ? 32 / NV : 1;   // lanes per score in the transposed layout
    static_assert(SB % (16 * 32) == 0 && R % KPW == 0, "attention stage shape");
    const int view = p.blk[l].view;
    const KView& vw = p.views[view];
    const int grp = p.Hq / p.Hkv;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int lg = lane / LPR, lr = lane % LPR;   // row group of the lane, lane within the row
    const int PSZ = attn_psz(grp, HD);

    unsigned char* myring = smem + warp * NST * SB;                   // [NST][SB] of this warp
    float* wo = reinterpret_cast<float*>(smem);                        // [kWarps][HG][HD], aliases the rings
    float* qs = reinterpret_cast<float*>(smem + RING);                 // [grp][HD] rotated queries
    float* wml = qs + grp * HD;                                        // [kWarps][HG][2] warp (m, l)
    float* wex = wml + kWarps * HG * 2;                                // [kWarps][HG] merge weights, [HG] maxima
    constexpr int PBS = (NV + HG + 3) & ~3;                            // floats per warp, 16-byte multiple
    float* wpb = qs + attn_pb_off(grp, HD, HG);                        // [kWarps][PBS] probabilities, rescales
    float* mypb = wpb + warp * PBS;
    const int cta = blockIdx.x;
    const bool eq = tab.cseg[view] > 0;
    const bool active = eq ? cta < p.B * p.Hkv * tab.cseg[view] : cta < tab.G[view];
    // the CTA's pieces: one (equal segments) or those of its position range
    const long long xbeg = active ? (eq ? 0 : attn_lo(tab, view, cta)) : 0;
    const long long xend = active ? (eq ? 1 : attn_lo(tab, view, cta + 1)) : 0;
    auto piece = [&](long long x, long long& nx) {
        if (eq) {
            nx = 1;
            return attn_piece_eq(p, vw, kv, tab, view, cta);
        }
        return attn_piece(p, vw, kv, tab, view, cta, x, nx);
    };
    const bool packed = vw.st == HD;   // consecutive ring slots are contiguous rows
    // keys and values stream evict-first, like the weights: the lines that phases
    // re-read (activations, partials, gains, prefetched weight boxes) keep their places
    const unsigned long long kvpol = l2_evict_first();
    bool any_split = false, aok = true;   // aok: warp-uniform, false once a stage wait of the warp gave up
    // earlier generic shared-memory accesses before the stage copies
    fence_proxy_async_smem();
    __syncthreads();

    for (long long x = xbeg, nx = 0; x < xend; x = nx) {
        const AttnPiece A = piece(x, nx);
        const int b = A.b, g = A.g;
        const int t_beg = A.t_beg, t_end = A.t_end;
        const KeyMap km = key_map(vw, kv[b]);
        const int nrounds = (t_end - t_beg + kWarps * R - 1) / (kWarps * R);
        const WT* kbase = reinterpret_cast<const WT*>(vw.k) + (long long)b * vw.sb + (long long)g * vw.sh;
        const WT* vbase = reinterpret_cast<const WT*>(vw.v) + (long long)b * vw.sb + (long long)g * vw.sh;

        // keys of round rd for this warp: [t0, t0 + cnt)
        auto slice_cnt = [&](int rd, int& t0) {
            t0 = t_beg + (rd * kWarps + warp) * R;
            const int c = t_end - t0;
            return rd < nrounds ? (c < 0 ? 0 : (c < R ? c : R)) : 0;
        };
        // lane 0: bulk copies of round rd's K and V rows into the warp's
        // stage rd % NST, one copy per run of consecutive ring slots when
        // rows are packed, completing on the stage barrier (nothing for an
        // empty slice: its stage is neither filled nor waited on; nothing
        // once a wait of the warp gave up)
        auto issue = [&](int rd) {
            int t0;
            const int cnt = slice_cnt(rd, t0);
            if (cnt > 0 && lane == 0 && aok) {
                const int si = rd % NST;
                unsigned char* buf = myring + si * SB;
                unsigned long long* bar = abar + warp * NST + si;
                mbar_arrive_expect_tx(bar, 2u * (unsigned int)cnt * RB);
                for (int r = 0; r < cnt;) {
                    const int slot = key_slot(km, t0 + r);
                    const int run = key_run(km, t0 + r, slot, packed ? cnt - r : 1);
                    bulk_g2s_pol(buf + r * RB, kbase + (long long)slot * vw.st, (unsigned int)(run * RB), bar, kvpol);
                    bulk_g2s_pol(buf + R * RB + r * RB, vbase + (long long)slot * vw.st, (unsigned int)(run * RB), bar,
                                 kvpol);
                    r += run;
                }
            }
        };

        for (int h0 = 0; h0 < grp; h0 += HG) {
            const int hn = grp - h0 < HG ? grp - h0 : HG;
            if (h0 == 0) {
                for (int r = 0; r + 1 < NST; ++r) issue(r);
                // q-norm + RoPE of the group's heads (warp h: head g * grp + h),
                // scaled by attn_scale; (cos, sin) of the position come from
                // the step's table
                if (warp < grp) {
                    constexpr int NQ = (HD / 8 + 31) / 32;   // float4 pairs per lane
                    // the query projection, or its split partials summed in order
                    const float* qraw = (p.tc_proj ? p.PB : p.QR) + (long long)b * p.QS + ((long long)g * grp + warp) * HD;
                    const int qS = p.tc_proj ? p.sk[PH_Q] : 1;
                    const long long qst = (long long)p.B * p.QS;
                    const float* gq = p.blk[l].q_norm;
                    const float4* cs = reinterpret_cast<const float4*>(
                        p.ROPEQ + ((long long)b * MTP_MAX_VIEWS + view) * (HD / 2));
                    float4 qa[NQ], qb[NQ], ga[NQ], gb[NQ], c0[NQ], c1[NQ];
                    float ss = 0.f;
#pragma unroll
                    for (int u = 0; u < NQ; ++u) {
                        const int i4 = lane + 32 * u;
                        if (i4 < HD / 8) {
                            qa[u] = __ldcg(reinterpret_cast<const float4*>(qraw) + i4);
                            qb[u] = __ldcg(reinterpret_cast<const float4*>(qraw + HD / 2) + i4);
                            ga[u] = __ldg(reinterpret_cast<const float4*>(gq) + i4);
                            gb[u] = __ldg(reinterpret_cast<const float4*>(gq + HD / 2) + i4);
                            c0[u] = __ldcg(cs + 2 * i4);
                            c1[u] = __ldcg(cs + 2 * i4 + 1);
                        }
                    }
                    if (qS > 1) {   // remaining split partials, after the first loads are in flight
#pragma unroll
                        for (int u = 0; u < NQ; ++u) {
                            const int i4 = lane + 32 * u;
                            if (i4 < HD / 8) {
                                const float4 a2 = ld4_sum(qraw + qst + 4 * i4, qS - 1, qst);
                                const float4 b2 = ld4_sum(qraw + qst + HD / 2 + 4 * i4, qS - 1, qst);
                                qa[u] = make_float4(qa[u].x + a2.x, qa[u].y + a2.y, qa[u].z + a2.z, qa[u].w + a2.w);
                                qb[u] = make_float4(qb[u].x + b2.x, qb[u].y + b2.y, qb[u].z + b2.z, qb[u].w + b2.w);
                            }
                        }
                    }
#pragma unroll
                    for (int u = 0; u < NQ; ++u) {
                        const int i4 = lane + 32 * u;
                        if (i4 < HD / 8) {
                            ss += qa[u].x * qa[u].x + qa[u].y * qa[u].y + qa[u].z * qa[u].z + qa[u].w * qa[u].w;
                            ss += qb[u].x * qb[u].x + qb[u].y * qb[u].y + qb[u].z * qb[u].z + qb[u].w * qb[u].w;
                        }
                    }
                    ss = warp_sum(ss);
                    const float rn = 1.0f / sqrtf(ss / (float)HD + p.eps);
                    float* qo = qs + warp * HD;
#pragma unroll
                    for (int u = 0; u < NQ; ++u) {
                        const int i4 = lane + 32 * u;
                        if (i4 < HD / 8) {
                            const float av[4] = {qa[u].x, qa[u].y, qa[u].z, qa[u].w};
                            const float bv[4] = {qb[u].x, qb[u].y, qb[u].z, qb[u].w};
                            const float gav[4] = {ga[u].x, ga[u].y, ga[u].z, ga[u].w};
                            const float gbv[4] = {gb[u].x, gb[u].y, gb[u].z, gb[u].w};
                            const float cv[4] = {c0[u].x, c0[u].z, c1[u].x, c1[u].z};
                            const float sv[4] = {c0[u].y, c0[u].w, c1[u].y, c1[u].w};
                            float ra[4], rb[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float a = av[e] * rn * gav[e];
                                const float c = bv[e] * rn * gbv[e];
                                ra[e] = (a * cv[e] - c * sv[e]) * p.attn_scale;
                                rb[e] = (a * sv[e] + c * cv[e]) * p.attn_scale;
                            }
                            reinterpret_cast<float4*>(qo)[i4] = make_float4(ra[0], ra[1], ra[2], ra[3]);
                            reinterpret_cast<float4*>(qo + HD / 2)[i4] = make_float4(rb[0], rb[1], rb[2], rb[3]);
                        }
                    }
                }
                __syncthreads();
            } else {
                __syncthreads();   // the previous pass's warp merge used the rings
                for (int r = 0; r + 1 < NST; ++r) issue(r);
            }

            // this lane's slice of the pass's queries
            float qr[HG][DPL];
#pragma unroll
            for (int hh = 0; hh < HG; ++hh)
#pragma unroll
                for (int c = 0; c < CPL; ++c)
#pragma unroll
                    for (int e4 = 0; e4 < EPC; e4 += 4) {
                        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                        if (hh < hn) v = *reinterpret_cast<const float4*>(qs + (h0 + hh) * HD + (c * LPR + lr) * EPC + e4);
                        qr[hh][c * EPC + e4 + 0] = v.x;
                        qr[hh][c * EPC + e4 + 1] = v.y;
                        qr[hh][c * EPC + e4 + 2] = v.z;
                        qr[hh][c * EPC + e4 + 3] = v.w;
                    }
            // online-softmax state: o for all HG heads on every lane; (m, l)
            // per head on every lane, or (transposed) of the lane's own head
            float o[HG][DPL];
            float m[TR ? 1 : HG], ls[TR ? 1 : HG];
#pragma unroll
            for (int hh = 0; hh < HG; ++hh)
#pragma unroll
                for (int d = 0; d < DPL; ++d) o[hh][d] = 0.f;
#pragma unroll
            for (int hh = 0; hh < (TR ? 1 : HG); ++hh) {
                m[hh] = -INFINITY;
                ls[hh] = 0.f;
            }

            for (int i = 0; i < nrounds && aok; ++i) {
                issue(i + NST - 1);   // its stage was consumed in round i - 1
                int t0;
                const int cnt = slice_cnt(i, t0);
                if (cnt > 0) {
                    const int si = i % NST;
                    if (!__all_sync(0xffffffffu, mbar_wait_limited(abar + warp * NST + si, (apar >> si) & 1u, p.timeout_ns))) {
                        // give up the pass: first wait (bounded again) for this
                        // round's and the issued later rounds' copies, so that
                        // none lands in shared memory afterwards
                        for (int r = i; r < i + NST && r < nrounds; ++r) {
                            int tr;
                            if (slice_cnt(r, tr) > 0)
                                mbar_wait_limited(abar + warp * NST + r % NST, (apar >> (r % NST)) & 1u, p.timeout_ns);
                        }
                        aok = false;
                        break;
                    }
                    apar ^= 1u << si;
                    const unsigned char* kb = myring + si * SB;
                    const unsigned char* vb = kb + R * RB;
                    float sc[NV];   // [RL][HG]
#pragma unroll
                    for (int x = 0; x < NV; ++x) sc[x] = 0.f;
#pragma unroll
                    for (int c = 0; c < CPL; ++c)
#pragma unroll
                        for (int ii = 0; ii < RL; ++ii) {
                            const uint4 w = *reinterpret_cast<const uint4*>(kb + (lg + KPW * ii) * RB + (c * LPR + lr) * 16);
#pragma unroll
                            for (int hh = 0; hh < HG; ++hh) sc[ii * HG + hh] += Chunk<WT>::dotr(w, &qr[hh][c * EPC]);
                        }
                    float pr[NV];   // probabilities of the round, [RL][HG]
                    float al[HG];   // rescale of the running o per head
                    if constexpr (TR) {
                        // lane holds score x = lane / SH: key x / HG, head x % HG
                        const float sx = transpose_sum<NV, 32>(sc);
                        const int x = lane / SH;
                        const bool valid = x / HG < cnt;
                        float mx = valid ? sx : -INFINITY;
#pragma unroll
                        for (int off = HG * SH; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
                        const float mn = fmaxf(m[0], mx);
                        const float mu = mn == -INFINITY ? 0.f : mn;
                        const float a = expf(m[0] - mu);
                        float pe = valid ? expf(sx - mu) : 0.f;
                        float ps = pe;
#pragma unroll
                        for (int off = HG * SH; off < 32; off <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
                        ls[0] = ls[0] * a + ps;
                        m[0] = mn;
                        if (lane % SH == 0) {
                            mypb[x] = pe;
                            if (x < HG) mypb[NV + x] = a;
                        }
                        __syncwarp();
                        if constexpr (NV % 4 == 0) {
#pragma unroll
                            for (int x4 = 0; x4 < NV; x4 += 4) {
                                const float4 v = *reinterpret_cast<const float4*>(mypb + x4);
                                pr[x4] = v.x;
                                pr[x4 + 1] = v.y;
                                pr[x4 + 2] = v.z;
                                pr[x4 + 3] = v.w;
                            }
                        } else {
#pragma unroll
                            for (int x4 = 0; x4 < NV; ++x4) pr[x4] = mypb[x4];
                        }
#pragma unroll
                        for (int hh = 0; hh < HG; ++hh) al[hh] = mypb[NV + hh];
                        __syncwarp();
                    } else {
#pragma unroll
                        for (int off = 1; off < LPR; off <<= 1)
#pragma unroll
                            for (int x = 0; x < NV; ++x) sc[x] += __shfl_xor_sync(0xffffffffu, sc[x], off);
#pragma unroll
                        for (int hh = 0; hh < HG; ++hh) {
                            float mx = -INFINITY;
#pragma unroll
                            for (int ii = 0; ii < RL; ++ii)
                                if (lg + KPW * ii < cnt) mx = fmaxf(mx, sc[ii * HG + hh]);
                            const float mn = fmaxf(m[hh], mx);
                            const float mu = mn == -INFINITY ? 0.f : mn;
                            al[hh] = expf(m[hh] - mu);
                            ls[hh] *= al[hh];
#pragma unroll
                            for (int ii = 0; ii < RL; ++ii) {
                                const float pe = lg + KPW * ii < cnt ? expf(sc[ii * HG + hh] - mu) : 0.f;
                                pr[ii * HG + hh] = pe;
                                ls[hh] += pe;
                            }
                            m[hh] = mn;
                        }
                    }
#pragma unroll
                    for (int hh = 0; hh < HG; ++hh)
#pragma unroll
                        for (int d = 0; d < DPL; ++d) o[hh][d] *= al[hh];
#pragma unroll
                    for (int c = 0; c < CPL; ++c)
#pragma unroll
                        for (int ii = 0; ii < RL; ++ii) {
                            if (lg + KPW * ii < cnt) {
                                const uint4 w = *reinterpret_cast<const uint4*>(vb + (lg + KPW * ii) * RB + (c * LPR + lr) * 16);
#pragma unroll
                                for (int e = 0; e < EPC; ++e) {
                                    const float v = Chunk<WT>::elem(w, e);
#pragma unroll
                                    for (int hh = 0; hh < HG; ++hh)
                                        o[hh][c * EPC + e] = fmaf(pr[ii * HG + hh], v, o[hh][c * EPC + e]);
                                }
                            }
                        }
                }
                __syncwarp();
            }

            // (m, l) of head hh for the warp state: transposed, from the lane
            // holding key 0 of head hh
            float mw[HG], lw[HG];
#pragma unroll
            for (int hh = 0; hh < HG; ++hh) {
                if constexpr (TR) {
                    mw[hh] = __shfl_sync(0xffffffffu, m[0], hh * SH);
                    lw[hh] = __shfl_sync(0xffffffffu, ls[0], hh * SH);
                } else {
                    mw[hh] = m[hh];
                    lw[hh] = ls[hh];
                }
            }
            // merge the row groups of the warp (rows of one round side by side)
#pragma unroll
            for (int off = LPR; off < 32; off <<= 1)
#pragma unroll
                for (int hh = 0; hh < HG; ++hh) {
                    const float m2 = __shfl_xor_sync(0xffffffffu, mw[hh], off);
                    const float l2 = __shfl_xor_sync(0xffffffffu, lw[hh], off);
                    const float mn = fmaxf(mw[hh], m2);
                    const float mu = mn == -INFINITY ? 0.f : mn;
                    const float a1 = expf(mw[hh] - mu), a2 = expf(m2 - mu);
                    lw[hh] = lw[hh] * a1 + l2 * a2;
#pragma unroll
                    for (int d = 0; d < DPL; ++d) {
                        const float o2 = __shfl_xor_sync(0xffffffffu, o[hh][d], off);
                        o[hh][d] = o[hh][d] * a1 + o2 * a2;
                    }
                    mw[hh] = mn;
                }
            __syncthreads();   // every warp is done with its ring
            if (lg == 0) {
#pragma unroll
                for (int hh = 0; hh < HG; ++hh) {
#pragma unroll
                    for (int c = 0; c < CPL; ++c)
#pragma unroll
                        for (int e4 = 0; e4 < EPC; e4 += 4)
                            *reinterpret_cast<float4*>(wo + (warp * HG + hh) * HD + (c * LPR + lr) * EPC + e4) =
                                make_float4(o[hh][c * EPC + e4], o[hh][c * EPC + e4 + 1], o[hh][c * EPC + e4 + 2],
                                            o[hh][c * EPC + e4 + 3]);
                    if (lr == 0) {
                        wml[(warp * HG + hh) * 2] = mw[hh];
                        wml[(warp * HG + hh) * 2 + 1] = lw[hh];
                    }
                }
            }
            __syncthreads();
            // CTA merge over the warps: weights per (warp, head), then the outputs
            if (tid < kWarps * HG) {
                const int hh = tid % HG;
                float M = -INFINITY;
#pragma unroll
                for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wml[(w * HG + hh) * 2]);
                wex[tid] = expf(wml[tid * 2] - (M == -INFINITY ? 0.f : M));
                if (tid < HG) wex[kWarps * HG + tid] = M;
            }
            __syncthreads();
            for (int oi = tid; oi < hn * HD; oi += kThreads) {
                const int hh = oi / HD, d = oi % HD;
                float Ls = 0.f, O = 0.f;
#pragma unroll
                for (int w = 0; w < kWarps; ++w) {
                    const float e = wex[w * HG + hh];
                    Ls = fmaf(e, wml[(w * HG + hh) * 2 + 1], Ls);
                    O = fmaf(e, wo[(w * HG + hh) * HD + d], O);
                }
                const int h = h0 + hh;
                if (A.S == 1) {
                    p.OB[((long long)b * p.Hq + (long long)g * grp + h) * HD + d] = O / Ls;
                } else {
                    float* part = p.PART + (long long)A.slot * PSZ;
                    part[h * HD + d] = O;
                    if (d == 0) {
                        part[grp * HD + h] = wex[kWarps * HG + hh];
                        part[grp * HD + grp + h] = Ls;
                    }
                }
            }
        }

        fence_proxy_async_smem();   // the merge's shared-memory writes before the next stage copies
        __syncthreads();
        if (A.S > 1 && !p.att_fold) {   // folded: the O prologue merges the partials after the barrier
            any_split = true;
            if (tid == 0) red_release_add(p.att_cnt + b * p.Hkv + g, 1u);
        }
    }
    if (!__syncthreads_and(aok)) {
        if (threadIdx.x == 0) atomicCAS(&p.hdr->status, 0, MTP_ERR_TIMEOUT);
        return false;
    }
    if (!any_split) return true;

    // merge: item s of an (b, g) with S items combines share s of the grp * HD
    // outputs over all S partials (lanes over partials, warps over outputs,
    // up to MJ outputs of a warp with their loads in flight together)
    constexpr int MJ = 4;
    constexpr int kMergeFew = 8;
    for (long long x = xbeg, nx = 0; x < xend; x = nx) {
        const AttnPiece A = piece(x, nx);
        if (A.S == 1) continue;
        if (!count_wait(p.att_cnt + A.b * p.Hkv + A.g, (unsigned int)A.S, p.hdr, p.timeout_ns)) return false;
        const int no = grp * HD;
        const int per = (no + A.S - 1) / A.S;
        const int o0 = (cta - A.cf) * per, o1 = o0 + per < no ? o0 + per : no;
        // the segment's first position (key-space partition)
        const long long s0 = eq ? 0 : x - A.t_beg;
        float* dst = p.OB + ((long long)A.b * p.Hq + (long long)A.g * grp) * HD;
        if (A.S <= kMergeFew) {
            // few partials: a thread per output, all its partials' loads in flight
            for (int j = o0 + (int)threadIdx.x; j < o1; j += kThreads) {
                const int h = j / HD;
                float mv[kMergeFew], lv[kMergeFew], ov[kMergeFew];
#pragma unroll
                for (int q = 0; q < kMergeFew; ++q) {
                    if (q < A.S) {
                        const float* pq = p.PART + (long long)attn_slot(tab, view, A.cf, q, s0) * PSZ;
                        mv[q] = __ldcg(pq + grp * HD + h);
                        lv[q] = __ldcg(pq + grp * HD + grp + h);
                        ov[q] = __ldcg(pq + j);
                    }
                }
                float M = -INFINITY;
#pragma unroll
                for (int q = 0; q < kMergeFew; ++q)
                    if (q < A.S) M = fmaxf(M, mv[q]);
                const float mu = M == -INFINITY ? 0.f : M;
                float Ls = 0.f, O = 0.f;
#pragma unroll
                for (int q = 0; q < kMergeFew; ++q) {
                    if (q < A.S) {
                        const float e = expf(mv[q] - mu);
                        Ls = fmaf(e, lv[q], Ls);
                        O = fmaf(e, ov[q], O);
                    }
                }
                dst[j] = O / Ls;
            }
            continue;
        }
        for (int j0 = o0 + warp; j0 < o1; j0 += MJ * kWarps) {
            float mm[MJ], ll[MJ], oo[MJ];
#pragma unroll
            for (int u = 0; u < MJ; ++u) { mm[u] = -INFINITY; ll[u] = 0.f; oo[u] = 0.f; }
            for (int q = lane; q < A.S; q += 32) {
                const float* pq = p.PART + (long long)attn_slot(tab, view, A.cf, q, s0) * PSZ;
                float mq[MJ], lq[MJ], oq[MJ];
#pragma unroll
                for (int u = 0; u < MJ; ++u) {
                    const int j = j0 + u * kWarps;
                    mq[u] = -INFINITY; lq[u] = 0.f; oq[u] = 0.f;
                    if (j < o1) {
                        mq[u] = __ldcg(pq + grp * HD + j / HD);
                        lq[u] = __ldcg(pq + grp * HD + grp + j / HD);
                        oq[u] = __ldcg(pq + j);
                    }
                }
#pragma unroll
                for (int u = 0; u < MJ; ++u) {
                    const float mn = fmaxf(mm[u], mq[u]);
                    const float mu = mn == -INFINITY ? 0.f : mn;
                    const float a1 = expf(mm[u] - mu), a2 = expf(mq[u] - mu);
                    ll[u] = ll[u] * a1 + lq[u] * a2;
                    oo[u] = oo[u] * a1 + oq[u] * a2;
                    mm[u] = mn;
                }
            }
#pragma unroll
            for (int u = 0; u < MJ; ++u) {
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) {
                    const float m2 = __shfl_xor_sync(0xffffffffu, mm[u], off);
                    const float l2 = __shfl_xor_sync(0xffffffffu, ll[u], off);
                    const float o2 = __shfl_xor_sync(0xffffffffu, oo[u], off);
                    const float mn = fmaxf(mm[u], m2);
                    const float mu = mn == -INFINITY ? 0.f : mn;
                    const float a1 = expf(mm[u] - mu), a2 = expf(m2 - mu);
                    ll[u] = ll[u] * a1 + l2 * a2;
                    oo[u] = oo[u] * a1 + o2 * a2;
                    mm[u] = mn;
                }
                const int j = j0 + u * kWarps;
                if (lane == 0 && j < o1) dst[j] = oo[u] / ll[u];
            }
        }
    }
    return true;
}

// The attention phase: out of line in the single-sequence kernel (its
// register allocation then does not compete with the GEMV phases'), inline
// in the batched kernel (measured faster there: 3.348 vs 3.396 ms per draft
// launch at 64 sequences, 1.650 vs 1.684 ms the other way at one sequence).
template <typename WT, int HD, int NST>
__device__ __noinline__ bool attention_call(const DraftParams& p, int l, unsigned char* smem, const int* kv,
                                            const AttnTab& tab, unsigned long long* abar, unsigned int& apar) {
    return attention_body<WT, HD, NST>(p, l, smem, kv, tab, abar, apar);
}
template <typename WT, int HD, int NST, bool TC>
__device__ __forceinline__ bool attention_phase(const DraftParams& p, int l, unsigned char* smem, const int* kv,
                                                const AttnTab& tab, unsigned long long* abar, unsigned int& apar) {
    if constexpr (TC) return attention_body<WT, HD, NST>(p, l, smem, kv, tab, abar, apar);
    else return attention_call<WT, HD, NST>(p, l, smem, kv, tab, abar, apar);
}

// ---------------------------------------------------------------------------
// LM head over the tied token table with the argmax folded in: per lane,
// per CTA in shared memory, then one atomic per sequence.
// One sequence: CTA c streams its block of rows [V c / grid, V (c + 1) /
// grid) with four groups of four warps; group q takes rows r0 + q, r0 + q + 4,
// ...  Every row is one bulk copy into one of the group's kHeadSlots
// shared-memory slots, so kHeadSlots rows per group are in flight.  The warps
// of a group split a row's chunks in quarters and hold their quarter of the
// input in registers; the group's first thread adds the four warp sums, runs
// the epilogue and refills the slot.  `par` carries the slot phase bits
// across calls.  False (status set) if a copy did not land in time.
__device__ __forceinline__ void group_sync(int g) {
    asm volatile("bar.sync %0, %1;" ::"r"(1 + g), "r"(kThreads / kHeadGroups) : "memory");
}

template <typename WT, int CPL>
__device__ bool head_groups_b1(const DraftParams& p, unsigned char* ring, unsigned long long (*bars)[kHeadSlots],
                               unsigned int& par, float (*hpart)[kHeadSlots][4], HeadEpi& e) {
    constexpr int EPC = Chunk<WT>::EPC;
    const WT* W = reinterpret_cast<const WT*>(p.tok_embd);
    const int nch = p.d_t / EPC, qch = (nch + 3) / 4;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int q = warp / 4, wq = warp % 4;
    const int r0 = row_lo(p.V, blockIdx.x), r1 = row_lo(p.V, blockIdx.x + 1);
    const int nrow = r1 - r0 > q ? (r1 - r0 - q + 3) / 4 : 0;
    const unsigned int rowb = (unsigned int)nch * 16u;
    unsigned char* gring = ring + q * kHeadSlots * p.head_slotb;
    const bool issuer = wq == 0 && lane == 0;
    float xr[CPL][EPC];
#pragma unroll
    for (int u = 0; u < CPL; ++u) {
        const int cw = lane + 32 * u, c = wq * qch + cw;
#pragma unroll
        for (int e4 = 0; e4 < EPC; e4 += 4) {
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (cw < qch && c < nch) v = __ldcg(reinterpret_cast<const float4*>(p.HN + c * EPC + e4));
            xr[u][e4] = v.x;
            xr[u][e4 + 1] = v.y;
            xr[u][e4 + 2] = v.z;
            xr[u][e4 + 3] = v.w;
        }
    }
    auto issue = [&](int j) {
        const int slot = j % kHeadSlots;
        mbar_arrive_expect_tx(&bars[q][slot], rowb);
        bulk_g2s_pol(gring + slot * p.head_slotb, W + (long long)(r0 + q + 4 * j) * nch * EPC, rowb, &bars[q][slot],
                     l2_evict_first());
    };
    __syncthreads();   // the slots reuse shared memory of earlier phases
    if (issuer) {
        fence_proxy_async_smem();
        for (int j = 0; j < kHeadSlots && j < nrow; ++j) issue(j);
    }
    for (int j = 0; j < nrow; ++j) {
        const int slot = j % kHeadSlots, bit = q * kHeadSlots + slot;
        if (!mbar_wait_limited(&bars[q][slot], (par >> bit) & 1u, p.timeout_ns)) {
            if (issuer) atomicCAS(&p.hdr->status, 0, MTP_ERR_TIMEOUT);
            for (int u = 1; u < kHeadSlots && j + u < nrow; ++u) {
                const int s2 = (j + u) % kHeadSlots;
                mbar_wait_limited(&bars[q][s2], (par >> (q * kHeadSlots + s2)) & 1u, p.timeout_ns);
            }
            return false;
        }
        par ^= 1u << bit;
        const unsigned char* sp = gring + slot * p.head_slotb;
        float acc = 0.f;
#pragma unroll
        for (int u = 0; u < CPL; ++u) {
            const int cw = lane + 32 * u, c = wq * qch + cw;
            if (cw < qch && c < nch) acc += Chunk<WT>::dotr(*reinterpret_cast<const uint4*>(sp + c * 16), xr[u]);
        }
        acc = warp_sum(acc);
        if (lane == 0) hpart[q][slot][wq] = acc;
        group_sync(q);   // the slot is consumed and the four sums are in
        if (issuer) {
            const float z[1] = {((hpart[q][slot][0] + hpart[q][slot][1]) + hpart[q][slot][2]) + hpart[q][slot][3]};
            e.apply(r0 + q + 4 * j, 0, 1, z, z);
            if (j + kHeadSlots < nrow) {
                fence_proxy_async_smem();
                issue(j + kHeadSlots);
            }
        }
    }
    return true;
}

// Tensor-core GEMM D[R, Bp] = W[R, K] X[Bp, K]^T (bf16, fp32 accumulate),
// with X split into bf16 high and low parts (two MMAs per K slice, so the
// product carries about 16 mantissa bits of X), or X taken as its high part.  Work items are (128-row
// tile, K split); CTA c takes items c, c + grid, ...  Warp 0 (one lane)
// streams the W and X tiles by tensor copies through a tc_stages-deep ring,
// warp 1 (one lane) issues the MMAs into one of two tensor-memory
// accumulators, and warps 4-7 read the accumulator (one tensor-memory lane
// per output row, 16 columns at a time) into the epilogue.  Barrier phases
// continue across calls through `ts`.
struct TcState {
    unsigned long long *full, *empty, *tfull, *tempty;
    unsigned int tmem;   // tensor-memory base address
    unsigned int g, it;  // K steps and items this CTA has processed so far
};

struct TcJob {
    const CUtensorMap *wa, *wb;   // W rows [0, R1) and [R1, R) (wb: rows counted from R1)
    const uint16_t *xh, *xl;      // X high / low parts, tiled (xtile_idx)
    int R1, R, nks, S, kps;       // rows, K steps of 64, K splits, K steps per split
    bool lo;                      // also multiply the low part (else X ~ its high part)
};

// The four epilogue warps (4-7) of tc_gemm synchronise among themselves.
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 5, 128;" ::: "memory"); }

template <class Epi>
__device__ __noinline__ bool tc_gemm(const DraftParams& p, const TcJob& J, unsigned char* smem, TcState& ts, Epi& epi) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int Bp = p.Bp, NS = p.tc_stages;
    const int ntiles = (J.R + kTcTileM - 1) / kTcTileM, nitems = ntiles * J.S;
    const int nit = nitems > (int)blockIdx.x ? (nitems - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
    const uint32_t abytes = kTcTileM * 128, xbytes = (uint32_t)Bp * 128, sbytes = abytes + 2 * xbytes;
    const uint32_t tx = abytes + (J.lo ? 2 : 1) * xbytes;       // bytes landing per stage
    const uint32_t base = (smem_addr(smem) + 1023u) & ~1023u;   // 1024-byte aligned ring
    unsigned char* ring = smem + (base - smem_addr(smem));
    auto ksteps = [&](int item, int& k0) {   // K steps of an item: [k0, k0 + n)
        k0 = (item % J.S) * J.kps;
        const int k1 = k0 + J.kps < J.nks ? k0 + J.kps : J.nks;
        return k1 - k0;
    };
    uint32_t nsteps = 0;   // K steps of this CTA's items (same on every thread)
    for (int j = 0; j < nit; ++j) {
        int k0;
        nsteps += (uint32_t)ksteps((int)blockIdx.x + j * (int)gridDim.x, k0);
    }
    bool ok = true;
    if (warp == 0) {
        if (lane == 0) {
            uint32_t g = ts.g;
            const unsigned long long pol = l2_evict_first();   // weight tiles: read once per step
            for (int j = 0; j < nit && ok; ++j) {
                const int item = (int)blockIdx.x + j * (int)gridDim.x;
                const int row0 = (item / J.S) * kTcTileM;
                const CUtensorMap* wm = row0 < J.R1 ? J.wa : J.wb;
                const int wy = row0 < J.R1 ? row0 : row0 - J.R1;
                int k0;
                const int n = ksteps(item, k0);
                // K steps in a rotated order per CTA, so the CTAs do not all
                // read the same shared X tile at once
                const int rot = n > 0 ? (int)blockIdx.x % n : 0;
                for (int i = 0; i < n; ++i, ++g) {
                    const int ks = k0 + (i + rot < n ? i + rot : i + rot - n);
                    const uint32_t st = g % NS;
                    if (!mbar_wait_limited(&ts.empty[st], ((g / NS) & 1u) ^ 1u, p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    unsigned char* sp = ring + st * sbytes;
                    mbar_arrive_expect_tx(&ts.full[st], tx);
                    tma_load_2d_pol(sp, wm, ks * kTcTileK, wy, &ts.full[st], pol);
                    bulk_g2s(sp + abytes, J.xh + (long long)ks * Bp * kTcTileK, xbytes, &ts.full[st]);
                    if (J.lo) bulk_g2s(sp + abytes + xbytes, J.xl + (long long)ks * Bp * kTcTileK, xbytes, &ts.full[st]);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            uint32_t g = ts.g;
            const uint32_t idesc = umma_idesc_bf16(kTcTileM, Bp);
            for (int j = 0; j < nit && ok; ++j) {
                const uint32_t it = ts.it + j, acc = it & 1u;
                if (!mbar_wait_limited(&ts.tempty[acc], ((it >> 1) & 1u) ^ 1u, p.timeout_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = ts.tmem + acc * (uint32_t)Bp;
                int k0;
                const int n = ksteps((int)blockIdx.x + j * (int)gridDim.x, k0);
                for (int ks = 0; ks < n; ++ks, ++g) {
                    const uint32_t st = g % NS;
                    if (!mbar_wait_limited(&ts.full[st], (g / NS) & 1u, p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = base + st * sbytes;
#pragma unroll
                    for (int kk = 0; kk < kTcTileK / 16; ++kk) {
                        const uint64_t ad = umma_desc_sw128(sa + kk * 32);
                        umma_bf16(d, ad, umma_desc_sw128(sa + abytes + kk * 32), idesc, (ks | kk) != 0 ? 1u : 0u);
                        if (J.lo) umma_bf16(d, ad, umma_desc_sw128(sa + abytes + xbytes + kk * 32), idesc, 1u);
                    }
                    umma_commit(&ts.empty[st]);
                }
                if (!ok) break;
                umma_commit(&ts.tfull[acc]);
            }
        }
    } else if (warp >= 4 && warp < 8) {
        // epilogue: accumulator -> shared-memory staging -> bulk stores (a
        // row segment per sequence), so the 128 threads issue a few copies
        // instead of one 4-byte store per value
        const int q = warp - 4;                  // tensor-memory lane quarter of this warp
        const int et = threadIdx.x - 4 * 32;     // 0..127
        const int r = 32 * q + lane;             // row of the tile this thread reads
        unsigned char* stg = ring + (size_t)NS * sbytes;
        for (int j = 0; j < nit && ok; ++j) {
            const uint32_t it = ts.it + j, acc = it & 1u;
            if (!mbar_wait_limited(&ts.tfull[acc], (it >> 1) & 1u, p.timeout_ns)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int item = (int)blockIdx.x + j * (int)gridDim.x;
            const int row0 = (item / J.S) * kTcTileM;
            if (j > 0) {   // the previous item's stores have read the staging
                bulk_wait_read();
                epi_sync();
            }
            const uint32_t ta = ts.tmem + ((uint32_t)(32 * q) << 16) + acc * (uint32_t)Bp;
            for (int c0 = 0; c0 < Bp; c0 += 16) {
                uint32_t v[16];
                tmem_ld16(ta + (uint32_t)c0, v);
                tmem_ld_wait();
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) epi.put(stg, row0, r, c0 + jj, __uint_as_float(v[jj]));
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ts.tempty[acc]);
            fence_proxy_async_smem();   // staging writes before the bulk copies read them
            epi_sync();
            epi.store(stg, row0, item % J.S, et);
            bulk_commit();
        }
        bulk_wait_all();              // the partials are written ...
        fence_proxy_async_global();   // ... and ordered before this thread's later generic accesses
    }
    ts.g += nsteps;
    ts.it += (uint32_t)nit;
    return __syncthreads_and(ok) != 0;
}

// LM head on tensor cores, step k: D[b, n] = sum_c h[b, c] E[n, c] over
// 256-row tiles of the token table E (tile t: rows 256 t ..), tile c,
// c + grid, ... on CTA c.  The batch block (kTcHeadM rows, zero past B) is
// the MMA's A operand and the table tile its B operand (M = 64, N = 256), so
// one MMA takes 8 KB of the table; with the table as the M side (M = 128,
// N = batch) the same loop issued twice the MMAs per byte and was bound by
// them.  Warp 0 (one lane) streams a 64 x 256 table box and the batch's
// bf16 block(s) of each K step through a th_stages-deep ring, warp 1 (one
// lane) issues the MMAs (greedy: h's high part; sampling: high and low)
// into one of two 256-column accumulators, and warps 4-7 read them back:
// accumulator row b lies in tensor-memory lane 32 (b / 16) + b % 16, so lane
// i < 16 of epilogue warp q owns sequence 16 q + i.  Each owner applies the
// softcap, stores the logits it is asked for, keeps its argmax key over its
// tiles and folds it into amax[k, b] once.  Barrier phases continue across
// steps through `ts` (a ring of its own: its stages differ from the
// projections').
// CONF: also keep each sequence's softmax denominator (the confidence
// output); a separate instantiation, so the plain head's epilogue loop
// carries none of it.
template <bool CONF>
static __device__ __noinline__ bool tc_head(const DraftParams& p, int k, unsigned char* smem, TcState& ts) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int NS = p.th_stages;
    const bool lo = p.sampling != 0;
    const uint32_t wbytes = kTcHeadN * 128, xbytes = kTcHeadM * 128;
    const uint32_t sbytes = wbytes + (lo ? 2 : 1) * xbytes;     // stage stride = bytes landing per stage
    const uint32_t tx = sbytes;
    const uint32_t base = (smem_addr(smem) + 1023u) & ~1023u;   // 1024-byte aligned ring
    unsigned char* ring = smem + (base - smem_addr(smem));
    const int ntiles = (p.V + kTcHeadN - 1) / kTcHeadN, nks = (p.d_t + kTcTileK - 1) / kTcTileK;
    const int nit = ntiles > (int)blockIdx.x ? (ntiles - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
    bool ok = true;
    if (warp == 0) {
        if (lane == 0) {
            uint32_t g = ts.g;
            const unsigned long long pol = l2_evict_first();   // the table: read once per step
            const int rot = (int)blockIdx.x % nks;               // K order rotated per CTA (the batch blocks are shared)
            for (int j = 0; j < nit && ok; ++j) {
                const int row0 = ((int)blockIdx.x + j * (int)gridDim.x) * kTcHeadN;
                for (int i = 0; i < nks; ++i, ++g) {
                    const int ks = i + rot < nks ? i + rot : i + rot - nks;
                    const uint32_t st = g % NS;
                    if (!mbar_wait_limited(&ts.empty[st], ((g / NS) & 1u) ^ 1u, p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    unsigned char* sp = ring + st * sbytes;
                    mbar_arrive_expect_tx(&ts.full[st], tx);
                    tma_load_2d_pol(sp, &p.tm_embd, ks * kTcTileK, row0, &ts.full[st], pol);
                    bulk_g2s(sp + wbytes, p.XH + (long long)ks * kTcHeadM * kTcTileK, xbytes, &ts.full[st]);
                    if (lo) bulk_g2s(sp + wbytes + xbytes, p.XL + (long long)ks * kTcHeadM * kTcTileK, xbytes, &ts.full[st]);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            uint32_t g = ts.g;
            const uint32_t idesc = umma_idesc_bf16(kTcHeadM, kTcHeadN);
            for (int j = 0; j < nit && ok; ++j) {
                const uint32_t it = ts.it + j, acc = it & 1u;
                if (!mbar_wait_limited(&ts.tempty[acc], ((it >> 1) & 1u) ^ 1u, p.timeout_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = ts.tmem + acc * (uint32_t)kTcHeadN;
                for (int ks = 0; ks < nks; ++ks, ++g) {
                    const uint32_t st = g % NS;
                    if (!mbar_wait_limited(&ts.full[st], (g / NS) & 1u, p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = base + st * sbytes;
#pragma unroll
                    for (int kk = 0; kk < kTcTileK / 16; ++kk) {
                        const uint64_t bd = umma_desc_sw128(sa + kk * 32);   // table tile, K slice kk
                        umma_bf16(d, umma_desc_sw128(sa + wbytes + kk * 32), bd, idesc, (ks | kk) != 0 ? 1u : 0u);
                        if (lo) umma_bf16(d, umma_desc_sw128(sa + wbytes + xbytes + kk * 32), bd, idesc, 1u);
                    }
                    umma_commit(&ts.empty[st]);
                }
                if (!ok) break;
                umma_commit(&ts.tfull[acc]);
            }
        }
    } else if (warp >= 4 && warp < 8) {
        const int q = warp - 4;   // tensor-memory lane quarter of this warp
        const int b = 16 * q + lane;
        const bool mine = lane < 16 && b < p.B;
        const int V = p.V;
        const float sc = p.softcap;
        float* const lg = p.out_logits ? p.out_logits + (long long)b * p.N * V + (long long)k * V : nullptr;
        float* const zb = p.ZB ? p.ZB + (long long)b * V : nullptr;
        // nothing to store, no softcap, no denominators: only the argmax
        const bool plain = !CONF && lg == nullptr && zb == nullptr && !(sc > 0.f);
        unsigned long long best = 0ull;
        SoftDen den = soft_den0();
        for (int j = 0; j < nit && ok; ++j) {
            const uint32_t it = ts.it + j, acc = it & 1u;
            if (!mbar_wait_limited(&ts.tfull[acc], (it >> 1) & 1u, p.timeout_ns)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int row0 = ((int)blockIdx.x + j * (int)gridDim.x) * kTcHeadN;
            const uint32_t ta = ts.tmem + ((uint32_t)(32 * q) << 16) + acc * (uint32_t)kTcHeadN;
            for (int c0 = 0; c0 < kTcHeadN; c0 += 32) {
                uint32_t ra[16], rb[16];   // two loads in flight, one wait
                tmem_ld16(ta + (uint32_t)c0, ra);
                tmem_ld16(ta + (uint32_t)c0 + 16u, rb);
                tmem_ld_wait();
                auto val = [&](int jj) { return __uint_as_float(jj < 16 ? ra[jj] : rb[jj - 16]); };
                if (!mine) continue;
                if (plain && row0 + c0 + 32 <= V) {
                    // the chunk's maximum by a tree, then its first position:
                    // the same key as the element-wise packed maximum (NaN
                    // only if all are NaN: key 0 at the first index; -0 and
                    // +0 compare equal)
                    float t[16];
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) t[jj] = fmaxf(val(jj), val(jj + 16));
#pragma unroll
                    for (int w = 8; w > 0; w >>= 1)
#pragma unroll
                        for (int jj = 0; jj < w; ++jj) t[jj] = fmaxf(t[jj], t[jj + w]);
                    const float m = t[0];
                    int ci = 0;
#pragma unroll
                    for (int jj = 31; jj >= 0; --jj) ci = val(jj) == m ? jj : ci;
                    const unsigned long long key = pack_argmax(m, (uint32_t)(row0 + c0 + ci));
                    best = key > best ? key : best;
                    continue;
                }
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    const int row = row0 + c0 + jj;
                    if (row < V) {
                        float z = val(jj);
                        if (sc > 0.f) z = sc * tanhf(z / sc);
                        if (lg) lg[row] = z;
                        if (zb) zb[row] = z;
                        const unsigned long long key = pack_argmax(z, (uint32_t)row);
                        best = key > best ? key : best;
                        if constexpr (CONF) den.add(z);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ts.tempty[acc]);
        }
        if (mine && nit > 0) atomicMax(p.amax + (long long)k * p.B + b, best);
        if (CONF && mine) p.CONF[(long long)blockIdx.x * p.B + b] = make_float2(den.m, den.s);
    }
    ts.g += (uint32_t)(nit * nks);
    ts.it += (uint32_t)nit;
    return __syncthreads_and(ok) != 0;
}

// epilogue: split partial of a projection, PB[split][b][row]
struct TcPartEpi {
    float* PB;
    int B, R;
    __device__ __forceinline__ void put(unsigned char* stg, int, int r, int b, float v) {
        reinterpret_cast<float*>(stg)[b * kTcTileM + r] = v;
    }
    // thread et < B stores sequence et's row segment
    __device__ __forceinline__ void store(const unsigned char* stg, int row0, int split, int et) {
        const int nr = R - row0 < kTcTileM ? R - row0 : kTcTileM;
        if (et < B && nr > 0)
            bulk_s2g(PB + ((long long)split * B + et) * R + row0, stg + (size_t)et * kTcTileM * 4, (unsigned)nr * 4u);
    }
};

// epilogue: unsplit post-projection: h, and its bf16 high / low parts as the
// head's operand (rows of the tile past R give zeros, so the operand's
// columns past d_t stay zero)
struct TcHnEpi {
    float* HN;
    uint16_t *XH, *XL;
    int B, R, Bp;
    __device__ __forceinline__ void put(unsigned char* stg, int row0, int r, int b, float v) {
        if (row0 + r >= R) v = 0.f;
        reinterpret_cast<float*>(stg)[b * kTcTileM + r] = v;
        const __nv_bfloat16 hi = __float2bfloat16_rn(v);
        const int kbl = r >> 6, kk = r & 63;
        const size_t o = (size_t)kbl * kTcHeadM * 128 + (size_t)b * 128 + (size_t)((((kk >> 3) ^ (b & 7)) << 3) | (kk & 7)) * 2;
        unsigned char* xs = stg + (size_t)kTcHeadM * kTcTileM * 4;
        *reinterpret_cast<uint16_t*>(xs + o) = __bfloat16_as_ushort(hi);
        *reinterpret_cast<uint16_t*>(xs + 2 * kTcHeadM * 128 + o) =
            __bfloat16_as_ushort(__float2bfloat16_rn(v - __bfloat162float(hi)));
    }
    // threads et < B store h's row segments; threads 64..67 the operand blocks
    __device__ __forceinline__ void store(const unsigned char* stg, int row0, int, int et) {
        const int nr = R - row0 < kTcTileM ? R - row0 : kTcTileM;
        if (et < B && nr > 0)
            bulk_s2g(HN + (long long)et * R + row0, stg + (size_t)et * kTcTileM * 4, (unsigned)nr * 4u);
        const int w = et - 64;
        if (w >= 0 && w < 4) {
            const int kbl = w & 1, kb = row0 / 64 + kbl;
            if (kb < (R + 63) / 64) {
                const unsigned char* xs = stg + (size_t)kTcHeadM * kTcTileM * 4 + (size_t)(w >> 1) * 2 * kTcHeadM * 128 +
                                          (size_t)kbl * kTcHeadM * 128;
                uint16_t* dst = ((w >> 1) ? XL : XH) + (long long)kb * Bp * 64;
                bulk_s2g(dst, xs, (unsigned)B * 128u);
            }
        }
    }
};

// job of projection phase `phase` of block l over the staged inputs
__device__ __forceinline__ TcJob tc_job(const DraftParams& p, int phase, int l) {
    TcJob J;
    J.xh = p.XA;
    J.xl = p.XAL;
    int K = 0;
    switch (phase) {
    case PH_PRE: J.wa = J.wb = &p.tm_w[0]; J.R = p.d_a; K = 2 * p.d_t; break;
    case PH_Q: J.wa = J.wb = &p.tm_w[2 + 5 * l]; J.R = p.QS; K = p.d_a; break;   // NextN: query, key and value rows
    case PH_O: J.wa = J.wb = &p.tm_w[2 + 5 * l + 1]; J.R = p.d_a; K = p.Hq * p.hd; break;
    case PH_FFN1: J.wa = &p.tm_w[2 + 5 * l + 2]; J.wb = &p.tm_w[2 + 5 * l + 3]; J.R = 2 * p.F; K = p.d_a; break;
    case PH_FFN2: J.wa = J.wb = &p.tm_w[2 + 5 * l + 4]; J.R = p.d_a; K = p.F; break;
    default: J.wa = J.wb = &p.tm_w[1]; J.R = p.d_t; K = p.d_a; break;   // PH_POST
    }
    J.R1 = phase == PH_FFN1 ? p.F : J.R;
    J.lo = true;
    J.nks = (K + kTcTileK - 1) / kTcTileK;
    J.S = p.sk[phase];
    J.kps = (J.nks + J.S - 1) / J.S;
    return J;
}

// L2 prefetch of this CTA's weight boxes of job J (thread 0, ahead of the
// phase's prologue and barrier: the weights do not depend on the phase's
// input, so their HBM latency hides behind the prologue)
__device__ __forceinline__ void tc_prefetch(const TcJob& J) {
    const int ntiles = (J.R + kTcTileM - 1) / kTcTileM, nitems = ntiles * J.S;
    for (int item = (int)blockIdx.x; item < nitems; item += (int)gridDim.x) {
        const int row0 = (item / J.S) * kTcTileM;
        const CUtensorMap* wm = row0 < J.R1 ? J.wa : J.wb;
        const int wy = row0 < J.R1 ? row0 : row0 - J.R1;
        const int k0 = (item % J.S) * J.kps, k1 = k0 + J.kps < J.nks ? k0 + J.kps : J.nks;
        for (int ks = k0; ks < k1; ++ks) tma_prefetch_2d(wm, ks * kTcTileK, wy);
    }
}

template <typename WT, bool TC>
__device__ __forceinline__ bool head_phase(const DraftParams& p, int k, const float* a, int lda,
                                           unsigned long long (*head_best)[32], unsigned char* smem,
                                           unsigned long long (*bars)[kHeadSlots], unsigned int& par,
                                           float (*hpart)[kHeadSlots][4], TcState& ts) {
    HeadEpi e{p.out_logits, p.V, p.N, k, p.softcap, 0ull, 0ull, p.ZB, p.out_conf != nullptr, soft_den0(), soft_den0()};
    if (TC && p.tc_head) {
        // greedy: h rounded to bf16 (half the MMAs and operand traffic; the
        // argmax is stable to it); sampling: both parts, so the sampler sees
        // logits as close as the CUDA-core path's.  The epilogue folds its
        // maxima into amax itself.
        if constexpr (TC) return p.out_conf ? tc_head<true>(p, k, smem, ts) : tc_head<false>(p, k, smem, ts);
        return false;
    } else if (p.head_slotb > 0) {
        const int cpl = (p.d_t / Chunk<WT>::EPC + 127) / 128;
        bool ok = true;
        switch (cpl) {
        case 1: ok = head_groups_b1<WT, 1>(p, smem, bars, par, hpart, e); break;
        case 2: ok = head_groups_b1<WT, 2>(p, smem, bars, par, hpart, e); break;
        case 3: ok = head_groups_b1<WT, 3>(p, smem, bars, par, hpart, e); break;
        case 4: ok = head_groups_b1<WT, 4>(p, smem, bars, par, hpart, e); break;
        default: ok = head_groups_b1<WT, 5>(p, smem, bars, par, hpart, e); break;
        }
        if (!__syncthreads_and(ok)) return false;
    } else {
        gemv<WT, 8, false>(reinterpret_cast<const WT*>(p.tok_embd), nullptr, p.V, p.d_t, a, lda, p.B, e,
                           &hpart[0][0][0]);   // the slots' partials are free here
    }
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
        if (e.conf) {   // the CTA's softmax-denominator partial of each column
            float* hm = reinterpret_cast<float*>(&head_best[0][0]);
            const SoftDen d = c0 == 0 ? e.den_lo : e.den_hi;
            hm[2 * (warp * 32 + lane)] = d.m;
            hm[2 * (warp * 32 + lane) + 1] = d.s;
            __syncthreads();
            if (threadIdx.x < 32 && c0 + (int)threadIdx.x < p.B) {
                SoftDen t = soft_den0();
                for (int w = 0; w < kWarps; ++w) t.merge(hm[2 * (w * 32 + threadIdx.x)], hm[2 * (w * 32 + threadIdx.x) + 1]);
                p.CONF[(long long)blockIdx.x * p.B + c0 + threadIdx.x] = make_float2(t.m, t.s);
            }
            __syncthreads();
        }
    }
    return true;
}

// ---------------------------------------------------------------------------
// centroid-routed LM head (Gemma 4 MTP page, sec. 3 "Centroid / ordered-
// embeddings LM head")
// ---------------------------------------------------------------------------
// Step k's logits over the candidates of each sequence's top_k centroids.
//   pass 1 (grid): CL[b, j] = centroids[j] . h_b over the n_c rows, and the
//     logit rows asked for (out_logits row (b, k), the sampler's ZB row b)
//     set to -1e30; a grid barrier.
//   pass 2 (no barrier): CTA c serves sequence b = c % B (b = c, c + G, ...
//     when the grid G is smaller than B).  It sorts b's n_c centroid keys
//     (value desc, id asc, NaN last) in shared memory, takes the first
//     top_k, and scores its share of their top_k * vsc candidates (centroid
//     j's list: the vsc ids at token_ordering[j vsc ...]):
//     z = softcap(tok_embd[t] . h_b), stored at t in the rows asked for,
//     folded into amax[k, b] and, with confidence, into the CTA's softmax
//     partial of b.  The CTAs serving one sequence each sort its keys (a few
//     microseconds) instead of meeting at a second barrier.
// An ordering entry outside [0, V) is skipped and sets the status to
// MTP_ERR_ARG.  Shared memory: (P + kRankSortMax) 8-byte keys (P = n_c
// rounded up to a power of two) and top_k ints.
template <typename WT>
static __device__ __noinline__ bool centroid_head(const DraftParams& p, int k, unsigned char* smem, float* red,
                                                  unsigned long long (*head_best)[32], unsigned int& epoch) {
    constexpr int EPC = Chunk<WT>::EPC, U = 4;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nc = p.n_cent, kc = p.cent_k, vsc = p.V / nc, B = p.B, G = (int)gridDim.x;
    const long long V = p.V;
    {
        StoreEpi e{p.CL, nc};
        gemv<WT, 8, false>(reinterpret_cast<const WT*>(p.cent), nullptr, nc, p.d_t, p.HN, p.d_t, B, e, red);
    }
    const long long nl = p.out_logits ? (long long)B * V : 0, nz = p.ZB ? (long long)B * V : 0;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < nl + nz; i += (long long)G * blockDim.x) {
        if (i < nl) {
            const long long b = i / V;
            p.out_logits[(b * p.N + k) * V + (i - b * V)] = -1e30f;
        } else {
            p.ZB[i - nl] = -1e30f;
        }
    }
    if (!grid_barrier(p.hdr, epoch, p.timeout_ns, G)) return false;

    unsigned int P = 1;
    while (P < (unsigned int)nc) P <<= 1;
    unsigned long long* keys = reinterpret_cast<unsigned long long*>(smem);
    unsigned long long* tmp = keys + P;
    int* sel = reinterpret_cast<int*>(tmp + kRankSortMax);
    if (p.out_conf)   // partials of the sequences this CTA does not serve stay empty
        for (int b = threadIdx.x; b < B; b += blockDim.x) p.CONF[(long long)blockIdx.x * B + b] = make_float2(-INFINITY, 0.f);
    const int nch = p.d_t / EPC, nrow = kc * vsc;
    const float sc = p.softcap;
    const unsigned long long pol = l2_evict_first();
    const bool wide = G >= B;
    for (int b = wide ? (int)blockIdx.x % B : (int)blockIdx.x; b < B; b += wide ? B : G) {
        const int gi = wide ? (int)blockIdx.x / B : 0, gn = wide ? (G - b + B - 1) / B : 1;
        const float* cl = p.CL + (long long)b * nc;
        __syncthreads();   // the previous sequence's keys and selection are consumed
        for (int j = threadIdx.x; j < nc; j += blockDim.x)
            keys[j] = ((unsigned long long)(~ordered_key(__ldcg(cl + j))) << 32) | (unsigned int)j;
        __syncthreads();
        sort_keys(keys, (unsigned int)nc, tmp);
        for (int r = threadIdx.x; r < kc; r += blockDim.x) sel[r] = (int)(keys[r] & 0xFFFFFFFFull);
        __syncthreads();
        const int lo = (int)((long long)nrow * gi / gn), hi = (int)((long long)nrow * (gi + 1) / gn);
        const float* h = p.HN + (long long)b * p.d_t;
        float* lg = p.out_logits ? p.out_logits + ((long long)b * p.N + k) * V : nullptr;
        float* zb = p.ZB ? p.ZB + (long long)b * V : nullptr;
        unsigned long long best = 0ull;
        SoftDen den = soft_den0();
        for (int r = lo + warp; r < hi; r += kWarps) {
            const int t = __ldg(p.cord + (long long)sel[r / vsc] * vsc + (r % vsc));
            if (t < 0 || (long long)t >= V) {
                if (lane == 0) atomicCAS(&p.hdr->status, 0, MTP_ERR_ARG);
                continue;
            }
            const uint4* wr = reinterpret_cast<const uint4*>(reinterpret_cast<const WT*>(p.tok_embd) + (long long)t * p.d_t);
            float acc = 0.f;
            for (int c0 = 0; c0 < nch; c0 += 32 * U) {
                uint4 w[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int c = c0 + lane + 32 * u;
                    w[u] = c < nch ? ld_weight16(wr + c, pol) : make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int c = c0 + lane + 32 * u;
                    if (c < nch) acc += Chunk<WT>::dot(w[u], h + c * EPC);
                }
            }
            float z = warp_sum(acc);   // every lane holds the row's logit
            if (sc > 0.f) z = sc * tanhf(z / sc);
            if (lane == 0) {
                if (lg) lg[t] = z;
                if (zb) zb[t] = z;
            }
            const unsigned long long key = pack_argmax(z, (uint32_t)t);
            best = key > best ? key : best;
            if (p.out_conf) den.add(z);
        }
        // the CTA's merge: one key and one softmax partial per warp
        float* hm = reinterpret_cast<float*>(&head_best[warp][1]);
        if (lane == 0) {
            head_best[warp][0] = best;
            hm[0] = den.m;
            hm[1] = den.s;
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            unsigned long long m = 0ull;
            SoftDen t = soft_den0();
            for (int w = 0; w < kWarps; ++w) {
                m = head_best[w][0] > m ? head_best[w][0] : m;
                const float* hw = reinterpret_cast<const float*>(&head_best[w][1]);
                t.merge(hw[0], hw[1]);
            }
            if (hi > lo) atomicMax(p.amax + (long long)k * B + b, m);
            if (p.out_conf) p.CONF[(long long)blockIdx.x * B + b] = make_float2(t.m, t.s);
        }
    }
    return true;
}

// Confidence of step k for sequence b (one warp): the top-1 softmax
// probability 1 / S, S the merged softmax denominator of the CTAs' partials
// (relative to their common maximum, the top logit).
__device__ __forceinline__ void write_conf(const DraftParams& p, int k, int b) {
    const int lane = threadIdx.x & 31;
    SoftDen t = soft_den0();
    for (int c = lane; c < (int)gridDim.x; c += 32) {
        const float2 v = __ldcg(p.CONF + (long long)c * p.B + b);
        t.merge(v.x, v.y);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, t.m, o), s2 = __shfl_xor_sync(0xffffffffu, t.s, o);
        t.merge(m2, s2);
    }
    if (lane == 0) p.out_conf[(long long)b * p.N + k] = t.s > 0.f ? 1.f / t.s : 0.f;
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
// Sampled drafting, step k: sample_dist over each sequence's logits
// (penalties over hist[b] and the drafts so far, temperature, min-p, top-p)
// and a draw with the uniform of (b, k, purpose 0): one pass of the
// sampler's pieces over the grid, the rows' finishing CTAs draw.  The token
// goes to the step's argmax slot, where the next step and the outputs read
// it; one grid barrier follows.
static __device__ __noinline__ bool sample_step(const DraftParams& p, int k, unsigned char* smem, unsigned int& epoch) {
    SampleJob j;
    j.base0 = p.ZB;
    j.base1 = nullptr;
    j.f32 = 1;
    j.mode = 1;
    j.B = p.B;
    j.N = p.N;
    j.V = p.V;
    j.draw_ld = p.V;
    j.draw_i = k;
    j.drafts = p.out_drafts;   // drafts 0..k-1 (written by the steps' PRE phases)
    j.drafts_ld = p.N;
    j.hist = p.hist;
    j.H = p.H;
    j.hist_ld = p.H;
    j.temp = p.s_temp;
    j.top_p = p.s_top_p;
    j.min_p = p.s_min_p;
    j.rep = p.s_rep;
    j.pres = p.s_pres;
    j.seed = p.seed;
    j.offset = p.offset;
    j.out_tokens = nullptr;
    j.out_n_accept = nullptr;
    j.out_draw = nullptr;
    j.out_draw_ld = 0;
    j.out_amax = p.amax + (long long)k * p.B;
    j.hdr = p.hdr;
    j.row_max = p.S_row;
    j.row_cnt = p.S_row + p.B;
    j.row_ovf = p.S_row + 2 * p.B;
    j.row_done = p.S_row + 3 * p.B;
    j.seq_done = nullptr;
    j.row_buf = p.S_buf;
    j.rcap = p.S_rcap;
    j.keep_id = nullptr;
    j.keep_w = nullptr;
    j.ccap = 0;
    j.n_keep = nullptr;
    j.w_keep = nullptr;
    j.piece_len = p.S_plen;
    j.ppr = p.S_ppr;
    j.next_piece = nullptr;   // static assignment: CTA c takes pieces c, c + grid, ...
    const int total = p.B * p.S_ppr;
    if (threadIdx.x == 0) prefetch_piece(j, blockIdx.x);
    for (int pc = blockIdx.x; pc < total; pc += gridDim.x)
        sample_piece(j, pc, pc + (int)gridDim.x < total ? pc + (int)gridDim.x : -1, smem);
    return grid_barrier(p.hdr, epoch, p.timeout_ns, gridDim.x);
}

// ---------------------------------------------------------------------------
// NextN: the drafter's own keys and values, and the block output
// ---------------------------------------------------------------------------

__device__ __forceinline__ void store_kv(float* d, float x) { *d = x; }
__device__ __forceinline__ void store_kv(uint16_t* d, float x) { *d = __bfloat16_as_ushort(__float2bfloat16_rn(x)); }

// Iteration k's key and value of every sequence with a row there, from the
// fused projection's key and value rows (QR, or on the tensor-core path its
// split-K partials summed in order): per KV head the key RMS-normed
// over hd with k_norm and rotated at the row position (NeoX pairs, the
// step's (cos, sin) table of view 0), both stored in the drafter's KV
// (views[0], slot = position) rounded to the weights' type.  A warp per
// (sequence, KV head), lanes over hd.  The attention reads these rows with
// bulk copies, so the writes are fenced for the async proxy; a grid barrier
// orders them before any read.
template <typename WT>
__device__ void nextn_kv_write(const DraftParams& p, int k, const int* kv) {
    const KView& vw = p.views[0];
    const int HD = p.hd, nh = HD / 2, lane = threadIdx.x & 31;
    const int nw = (int)gridDim.x * kWarps;
    for (int it = (int)blockIdx.x * kWarps + (int)(threadIdx.x >> 5); it < p.B * p.Hkv; it += nw) {
        const int b = it / p.Hkv, g = it - b * p.Hkv;
        if (k < 0 && catchup_row(p, b, k) < 0) continue;   // no catch-up row of b at this iteration
        const long long pos = row_pos(p, kv, b, k);
        // the projection's key and value rows: QR, or the split-K partials summed in order
        const float* src = (p.tc_proj ? p.PB : p.QR) + (long long)b * p.QS;
        const int S = p.tc_proj ? p.sk[PH_Q] : 1;
        const long long st = (long long)p.B * p.QS;
        auto raw = [&](int off) {
            float v = __ldcg(src + off);
            for (int s = 1; s < S; ++s) v += __ldcg(src + s * st + off);
            return v;
        };
        const int ko = (p.Hq + g) * HD, vo = (p.Hq + p.Hkv + g) * HD;
        float ss = 0.f;
        for (int d = lane; d < HD; d += 32) {
            const float x = raw(ko + d);
            ss = fmaf(x, x, ss);
        }
        ss = warp_sum(ss);
        const float rn = 1.0f / sqrtf(ss / (float)HD + p.eps);
        const float* gk = p.blk[0].k_norm;
        const float2* cs = p.ROPEQ + (long long)b * MTP_MAX_VIEWS * nh;   // view 0
        WT* kd = reinterpret_cast<WT*>(const_cast<void*>(vw.k)) + (long long)b * vw.sb + (long long)g * vw.sh + pos * vw.st;
        WT* vd = reinterpret_cast<WT*>(const_cast<void*>(vw.v)) + (long long)b * vw.sb + (long long)g * vw.sh + pos * vw.st;
        for (int i = lane; i < nh; i += 32) {
            const float a = raw(ko + i) * rn * __ldg(gk + i);
            const float c = raw(ko + nh + i) * rn * __ldg(gk + nh + i);
            const float2 t = __ldcg(cs + i);   // (cos, sin)
            store_kv(kd + i, a * t.x - c * t.y);
            store_kv(kd + nh + i, a * t.y + c * t.x);
        }
        for (int d = lane; d < HD; d += 32) store_kv(vd + d, raw(vo + d));
    }
    fence_proxy_async_global();
}

// The block output h' = x_m + y2 of every sequence (no post-norm, no
// projection; y2 the down projection, or on the tensor-core path its split-K
// partials summed in order): HX, the next step's hidden state, and HN =
// head_norm(h'), the LM head's input (with the tensor-core head also as the
// head operand's bf16 high and low parts).  CTA c takes sequences c,
// c + grid, ...
static __device__ void nextn_post(const DraftParams& p, float* x, float* gs, float* dst, float* red) {
    const int n = p.d_t;
    const int S = p.tc_proj ? p.sk[PH_FFN2] : 1;
    const float* y2 = p.tc_proj ? p.PB : p.Y2;
    const long long st = (long long)p.B * n;
    for (int b = blockIdx.x; b < p.B; b += gridDim.x) {
        for (int i = threadIdx.x; i < n; i += blockDim.x) {
            float y = __ldcg(y2 + (long long)b * n + i);
            for (int s = 1; s < S; ++s) y += __ldcg(y2 + s * st + (long long)b * n + i);
            const float v = __ldcg(p.XM + (long long)b * n + i) + y;
            x[i] = v;
            p.HX[(long long)b * n + i] = v;
            gs[i] = __ldg(p.final_norm + i);
        }
        __syncthreads();
        rms_into_s(x, gs, n, p.eps, dst, red);
        for (int i = threadIdx.x; i < n; i += blockDim.x) {
            const float v = dst[i];
            p.HN[(long long)b * n + i] = v;
            if (p.tc_head) {
                const long long xi = xtile_idx(b, i, kTcHeadM);
                const __nv_bfloat16 hi = __float2bfloat16_rn(v);
                p.XH[xi] = __bfloat16_as_ushort(hi);
                p.XL[xi] = __bfloat16_as_ushort(__float2bfloat16_rn(v - __bfloat162float(hi)));
            }
        }
        __syncthreads();
    }
    if (p.tc_head) fence_proxy_async_global();   // the head operand is read by bulk copies
}

// PT: the projections' weight type (WT, or int8_t / Q4Code for Q8_0 / Q4_0 codes with block scales)
template <typename WT, int HD, bool TC, typename PT>
__device__ __forceinline__ void draft_body(const DraftParams& p, unsigned char* smem, TcState& ts, TcState& hs) {
    __shared__ float red[2 * kWarps];
    __shared__ unsigned long long head_best[kWarps][32];
    __shared__ __align__(8) unsigned long long head_bar[kHeadGroups][kHeadSlots];   // LM head slots
    __shared__ float head_part[kHeadGroups][kHeadSlots][4];
    unsigned int head_par = 0;
    __shared__ __align__(8) unsigned long long attn_bar[kWarps][kAttnStagesTc];   // attention stage barriers
    unsigned int attn_par = 0;
    unsigned int epoch = 0;
    float* tmp = reinterpret_cast<float*>(smem);                 // [max(d_a)] residual scratch
    float* act = tmp + ((p.d_a + 3) & ~3);                       // activations
    constexpr int U = 8;
    bool ok = true;

    // device-side input checks: every CTA evaluates the same predicate, so on
    // bad inputs all CTAs return before the first barrier
    {
        bool bad = false;
        for (int b = 0; b < p.B; ++b) {
            const int kl = p.kv_len[b], tk = p.last_tok[b];
            if (kl < (p.nextn ? 0 : 1) || tk < 0 || tk >= p.V) bad = true;
            if (p.nextn) {
                // the drafter's KV must hold every row this call writes
                const int nc = p.n_cu ? p.n_cu[b] : 0;
                if (nc < 0 || nc > p.M || (long long)kl + nc + p.N > p.views[0].cap) bad = true;
                for (int j = 0; j < nc && !bad; ++j) {
                    const int t = p.cu_tok[(long long)b * p.M + j];
                    if (t < 0 || t >= p.V) bad = true;
                }
                continue;
            }
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
    // tensor-core head: zero rows B..Bp-1 of the bf16 parts of h (read by
    // tensor copies, first after >= 1 barrier)
    // tensor-core operands: zero once (rows >= B and columns past a row's
    // length are never written; bulk copies read them from the first phase
    // on, after >= 1 barrier)
    if (TC && p.tc_head) {
        const long long nh = (long long)((p.d_t + 63) / 64) * kTcHeadM * 64,
                        na = p.tc_proj ? (long long)((p.kmax + 63) / 64) * p.Bp * 64 : 0;
        for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < 2 * nh + 2 * na;
             i += (long long)gridDim.x * blockDim.x) {
            if (i < nh) p.XH[i] = 0;
            else if (i < 2 * nh) p.XL[i - nh] = 0;
            else if (i < 2 * nh + na) p.XA[i - 2 * nh] = 0;
            else p.XAL[i - 2 * nh - na] = 0;
        }
        fence_proxy_async_global();
    }
    // sequence lengths, read once, and the attention item tables
    __shared__ int s_kv[MTP_MAX_BATCH];
    __shared__ int s_kx[MTP_MAX_BATCH];   // NextN: keys of the current draft step
    __shared__ AttnTab s_tab;
    for (int b = threadIdx.x; b < p.B; b += blockDim.x) s_kv[b] = p.kv_len[b];
    __syncthreads();
    attn_tab_fill(p, s_kv, attn_geom(HD, (int)sizeof(WT)).R, s_tab);
    __syncthreads();
    // RoPE inverse frequencies theta^(-2i/hd) of every view, in fp64, spread
    // over the grid (first read after the first barrier)
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < MTP_MAX_VIEWS * (HD / 2); e += gridDim.x * blockDim.x) {
        const float th = p.views[e / (HD / 2)].theta;
        p.ROPE[e] = th > 0.f ? exp(-2.0 * (double)(e % (HD / 2)) / (double)HD * log((double)th)) : 0.0;
    }

    if (threadIdx.x < kHeadGroups * kHeadSlots) mbar_init(&head_bar[0][0] + threadIdx.x, 1);
    if (threadIdx.x < kWarps * kAttnStagesTc) mbar_init(&attn_bar[0][0] + threadIdx.x, 1);
    mbar_fence_init();
    __syncthreads();
    // one GEMV phase and the barrier after it
    auto gemv_step = [&](int phase, int k, int l, const void* W, const void* W2, const uint16_t* S,
                         const uint16_t* S2, int R, int K, auto& epi, auto two) -> bool {
        constexpr bool TWO = decltype(two)::value;
        int lda = 0;
        bool ok = true;
        if constexpr (TC) {
            if (p.tc_proj && threadIdx.x == 0) tc_prefetch(tc_job(p, phase, l));
        }
        const float* a = stage_act<WT, TC>(p, phase, k, l, act, tmp, red, epoch, lda, ok, &s_tab);
        if (!ok) return false;
        if (TC && p.tc_proj) {
            // tensor cores over the staged bf16 input parts: split partials,
            // or (post-projection, unsplit) h and its bf16 parts for the head
            if constexpr (TC) {
                const TcJob J = tc_job(p, phase, l);
                if (phase == PH_POST) {
                    TcHnEpi he{p.HN, p.XH, p.XL, p.B, p.d_t, kTcHeadM};
                    if (!tc_gemm(p, J, smem, ts, he)) return false;
                } else {
                    TcPartEpi pe{p.PB, p.B, J.R};
                    if (!tc_gemm(p, J, smem, ts, pe)) return false;
                }
            }
        } else {
            gemv<PT, TWO ? U / 2 : U, TWO>(reinterpret_cast<const PT*>(W), reinterpret_cast<const PT*>(W2), R, K, a,
                                           lda, p.B, epi, red, S, S2);
        }
        if (TC && p.tc_head && phase == PH_POST) fence_proxy_async_global();   // h parts are read by tensor copies
        return grid_barrier(p.hdr, epoch, p.timeout_ns, gridDim.x);
    };
    using One = std::integral_constant<bool, false>;
    using Two = std::integral_constant<bool, true>;

    // NextN: iterations -C .. -1 are the catch-up rows, C the largest count
    // of any sequence (PRE, then the key and value rows of Q and their
    // store); 0 .. N-1 the draft steps.  Every CTA reads the same counts.
    int k0 = 0;
    if (p.nextn && p.n_cu)
        for (int b = 0; b < p.B; ++b) k0 = max(k0, __ldg(p.n_cu + b));
    for (int k = -k0; k < p.N; ++k) {
        // ---- PRE ----
        if (blockIdx.x == 0) {
            for (int b = threadIdx.x; b < p.B; b += blockDim.x) {
                if (k > 0) p.out_drafts[(long long)b * p.N + (k - 1)] = step_token(p, b, k);
            }
        }
        if (k > 0 && p.out_conf)   // the previous step's confidence, a warp per sequence
            for (int b = blockIdx.x * kWarps + (int)(threadIdx.x >> 5); b < p.B; b += gridDim.x * kWarps)
                write_conf(p, k - 1, b);
        {
            StoreEpi e{p.XB, p.d_a};
            if (!gemv_step(PH_PRE, k, 0, p.w_pre, nullptr, p.s_pre, nullptr, p.d_a, 2 * p.d_t, e, One{})) return;
        }

        for (int l = 0; l < p.L; ++l) {
            const BlkW& bw = p.blk[l];
            // ---- Q ----
            if (l == 0) {
                // (cos, sin) of this step's query position for every sequence
                // and view: angle in fp64, reduced to [-pi, pi] before the
                // fp32 sin/cos (first read after the Q barrier)
                constexpr int nh = HD / 2;
                for (int e = threadIdx.x * gridDim.x + blockIdx.x; e < p.B * MTP_MAX_VIEWS * nh;
                     e += gridDim.x * blockDim.x) {
                    const double f = __ldcg(p.ROPE + e % (MTP_MAX_VIEWS * nh));
                    if (f > 0.0) {
                        double ang = (double)row_pos(p, s_kv, e / (MTP_MAX_VIEWS * nh), k) * f;
                        ang -= 6.283185307179586 * rint(ang * 0.15915494309189535);
                        float sn, cs;
                        sincosf((float)ang, &sn, &cs);
                        p.ROPEQ[e] = make_float2(cs, sn);
                    }
                }
            }
            if (!p.nextn) {
                StoreEpi e{p.QR, p.QS};
                if (!gemv_step(PH_Q, k, l, bw.w_q, nullptr, bw.s_q, nullptr, p.Hq * p.hd, p.d_a, e, One{})) return;
            } else {
                // ---- QKV (NextN): the fused projection; a catch-up row needs its key and value rows only ----
                // (the tensor-core path runs the whole projection for a catch-up row too)
                const int q0 = k < 0 && !p.tc_proj ? p.Hq * p.hd : 0;
                StoreEpi e{p.QR + q0, p.QS};
                if (!gemv_step(PH_Q, k, l, weight_rows(reinterpret_cast<const PT*>(bw.w_q), q0, p.d_a), nullptr,
                               bw.s_q ? bw.s_q + (long long)q0 * (p.d_a / 32) : nullptr, nullptr, p.QS - q0, p.d_a, e,
                               One{}))
                    return;
                nextn_kv_write<WT>(p, k, s_kv);
                if (k < 0) break;   // catch-up: the next PRE's barrier orders the stores
                if (!grid_barrier(p.hdr, epoch, p.timeout_ns, gridDim.x)) return;
                // this step's keys: the rows before it, the catch-up rows, the steps so far and its own
                for (int b = threadIdx.x; b < p.B; b += blockDim.x)
                    s_kx[b] = s_kv[b] + (p.n_cu ? __ldg(p.n_cu + b) : 0) + k + 1;
                __syncthreads();
                attn_tab_fill(p, s_kx, attn_geom(HD, (int)sizeof(WT)).R, s_tab);
                __syncthreads();
            }
            // ---- ATT ----
            if (!attention_phase<WT, HD, TC ? kAttnStagesTc : kAttnStages, TC>(p, l, smem, p.nextn ? s_kx : s_kv,
                                                                              s_tab, &attn_bar[0][0], attn_par))
                return;
            if (!grid_barrier(p.hdr, epoch, p.timeout_ns, gridDim.x)) return;
            // every CTA has passed its attention waits: reset the item counters
            if (blockIdx.x == 0)
                for (int i = threadIdx.x; i < p.B * p.Hkv; i += blockDim.x) p.att_cnt[i] = 0u;
            // ---- O ----
            {
                StoreEpi e{p.YB, p.d_a};
                if (!gemv_step(PH_O, k, l, bw.w_o, nullptr, bw.s_o, nullptr, p.d_a, p.Hq * p.hd, e, One{})) return;
            }
            // ---- FFN1 (gate and up share the input; GeGLU in the epilogue) ----
            {
                GegluEpi e{p.MB, p.F, p.nextn};
                if (!gemv_step(PH_FFN1, k, l, bw.w_gate, bw.w_up, bw.s_gate, bw.s_up, p.F, p.d_a, e, Two{})) return;
            }
            // ---- FFN2 ----
            {
                StoreEpi e{p.Y2, p.d_a};
                if (!gemv_step(PH_FFN2, k, l, bw.w_down, nullptr, bw.s_down, nullptr, p.d_a, p.F, e, One{})) return;
            }
        }
        if (k < 0) continue;   // NextN catch-up iteration: done after its key and value
        // ---- POST ----
        if (p.nextn) {
            nextn_post(p, tmp, act + p.kmax, act, red);
            if (!grid_barrier(p.hdr, epoch, p.timeout_ns, gridDim.x)) return;
        } else if (TC && p.tc_head) {
            StoreXhEpi e{p.HN, p.d_t, p.XH, p.XL, kTcHeadM};
            if (!gemv_step(PH_POST, k, 0, p.w_post, nullptr, p.s_post, nullptr, p.d_t, p.d_a, e, One{})) return;
        } else {
            StoreEpi e{p.HN, p.d_t};
            if (!gemv_step(PH_POST, k, 0, p.w_post, nullptr, p.s_post, nullptr, p.d_t, p.d_a, e, One{})) return;
        }
        // ---- HEAD ----
        if (p.n_cent > 0) {
            if (!centroid_head<WT>(p, k, smem, red, head_best, epoch)) return;
        } else {
            int lda = 0;
            const float* a = nullptr;
            if (p.head_slotb == 0 && !(TC && p.tc_head)) {
                a = stage_act<WT, TC>(p, PH_HEAD, k, 0, act, tmp, red, epoch, lda, ok, &s_tab);
                if (!ok) return;
            }
            if (!head_phase<WT, TC>(p, k, a, lda, head_best, smem, head_bar, head_par, head_part, hs)) return;
        }
        if (!grid_barrier(p.hdr, epoch, p.timeout_ns, gridDim.x)) return;
        // ---- SAMPLE (temperature > 0): sample_dist of the step's logits ----
        if (p.sampling && !sample_step(p, k, smem, epoch)) return;
    }
    // outputs of the last step
    if (p.out_conf)
        for (int b = blockIdx.x * kWarps + (int)(threadIdx.x >> 5); b < p.B; b += gridDim.x * kWarps)
            write_conf(p, p.N - 1, b);
    if (blockIdx.x == 0) {
        for (int b = threadIdx.x; b < p.B; b += blockDim.x)
            p.out_drafts[(long long)b * p.N + (p.N - 1)] = step_token(p, b, p.N);
        if (p.out_h_last)
            for (long long i = threadIdx.x; i < (long long)p.B * p.d_t; i += blockDim.x)
                p.out_h_last[i] = __ldcg((p.nextn ? p.HX : p.HN) + i);
    }
}

// The persistent draft kernel.  TC: the variant with the tensor-core paths,
// whose tensor memory is allocated by warp 2 before the body and freed after
// it; every exit of the body is uniform over the CTA.
template <typename WT, int HD, bool TC, typename PT>
__global__ void __launch_bounds__(kThreads, 1) draft_kernel(const __grid_constant__ DraftParams p) {
    extern __shared__ __align__(16) unsigned char smem[];
    constexpr int NB = 2 * kTcMaxStages + 4;   // barriers of one ring
    __shared__ __align__(8) unsigned long long tc_bar[2 * NB];   // the projections' ring, then the head's
    __shared__ unsigned int tc_tmem;
    TcState ts{tc_bar, tc_bar + kTcMaxStages, tc_bar + 2 * kTcMaxStages, tc_bar + 2 * kTcMaxStages + 2, 0u, 0u, 0u};
    unsigned long long* hb = tc_bar + NB;
    TcState hs{hb, hb + kTcMaxStages, hb + 2 * kTcMaxStages, hb + 2 * kTcMaxStages + 2, 0u, 0u, 0u};
    const int warp = threadIdx.x >> 5;
    if (TC && p.tc_head) {
        // per ring: full / empty stage barriers (one arrival each),
        // accumulator full (one commit) and empty (one arrival per epilogue
        // warp)
        if (threadIdx.x < 2 * NB)
            mbar_init(&tc_bar[threadIdx.x], threadIdx.x % NB >= 2 * kTcMaxStages + 2 ? 4u : 1u);
        if (warp == 2) {
            tmem_alloc(&tc_tmem, (unsigned int)p.tc_cols);
            tmem_relinquish();
        }
        mbar_fence_init();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        ts.tmem = tc_tmem;
        hs.tmem = tc_tmem;
    }
    draft_body<WT, HD, TC, PT>(p, smem, ts, hs);
    if (TC && p.tc_head) {
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (warp == 2) tmem_dealloc(ts.tmem, (unsigned int)p.tc_cols);
    }
}

template <typename WT, int HD, bool TC, typename PT = WT>
cudaError_t launch_draft_t(const DraftParams& p, int grid, size_t smem, cudaStream_t s) {
    cudaError_t e =
        cudaFuncSetAttribute(draft_kernel<WT, HD, TC, PT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    void* args[] = {const_cast<DraftParams*>(&p)};
    return cudaLaunchCooperativeKernel((const void*)draft_kernel<WT, HD, TC, PT>, dim3(grid), dim3(kThreads), args,
                                       smem, s);
}

template <typename WT, int HD, bool TC, typename PT = WT>
int draft_blocks_per_sm_t(size_t smem) {
    int n = 0;
    cudaFuncSetAttribute(draft_kernel<WT, HD, TC, PT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, draft_kernel<WT, HD, TC, PT>, kThreads, smem) !=
        cudaSuccess)
        return 0;
    return n;
}

}  // namespace mtp
