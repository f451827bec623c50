// sample.cuh -- sample_dist on the GPU ("opus-mtp-turbo: Track 1 report",
// item 4: penalties over history + window inputs, temperature, min-p, top-p;
// exact speculative acceptance and the residual max(p - q, 0)).
//
// The sampler's arithmetic decides integers, so every step is IEEE fp32 with
// its rounding written out (no contraction): penalised logit z / r or z * r,
// minus the presence penalty, divided by the temperature; weight
// w = exp(l - lmax); every sum runs sequentially in (w desc, id asc) order.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "verify.cuh"

namespace mtp {

// exp(x) for x <= 0 in fp32 (Cody and Waite 1980: x = k ln2 + r with ln2
// split into a 16-bit head and a tail so k * head is exact; exp(r) on
// |r| <= ln2 / 2 by its Taylor series through r^7 in Horner form with fused
// multiply-adds; scaled by 2^k).  0 below -87.
__device__ __forceinline__ float exp_cw(float x) {
    if (!(x >= -87.0f)) return 0.0f;
    const float k = rintf(__fmul_rn(x, 1.44269504088896341f));
    float r = __fmaf_rn(-k, 0.693145751953125f, x);
    r = __fmaf_rn(-k, 1.42860682030941723e-06f, r);
    float q = 1.0f / 5040.0f;
    q = __fmaf_rn(q, r, 1.0f / 720.0f);
    q = __fmaf_rn(q, r, 1.0f / 120.0f);
    q = __fmaf_rn(q, r, 1.0f / 24.0f);
    q = __fmaf_rn(q, r, 1.0f / 6.0f);
    q = __fmaf_rn(q, r, 0.5f);
    q = __fmaf_rn(q, r, 1.0f);
    q = __fmaf_rn(q, r, 1.0f);
    const int ki = (int)k;  // -126 <= ki <= 0
    return __fmul_rn(q, __int_as_float((ki + 127) << 23));
}

// penalised, temperature-scaled logit
__device__ __forceinline__ float scaled_logit(const VerifySampleArgs& a, float z, bool pen) {
    float y = z;
    if (pen) {
        y = z > 0.f ? __fdiv_rn(z, a.rep) : __fmul_rn(z, a.rep);
        y = __fsub_rn(y, a.pres);
    }
    return __fdiv_rn(y, a.temp);
}

// Row geometry: rows [0, B(1+N)) are target rows (b, i), rows [B(1+N),
// B(1+N) + B N) are draft rows (b, i); in draft sampling (draft_k >= 0) row
// b is sequence b at step draft_k.  Penalty set of (b, i): hist[b][*] u
// drafts[b][0..i-1].
struct RowInfo {
    const void* base;
    int b, i;
};

__device__ __forceinline__ RowInfo row_info(const VerifySampleArgs& a, int row) {
    RowInfo r;
    const int R = a.N + 1;
    const long long esz = a.bf16 ? 2 : 4;
    if (a.draft_k >= 0) {   // draft sampling: one row per sequence, tgt = [B, V]
        r.b = row;
        r.i = a.draft_k;
        r.base = static_cast<const char*>(a.tgt) + (long long)row * a.V * esz;
    } else if (row < a.B * R) {
        r.b = row / R;
        r.i = row % R;
        r.base = static_cast<const char*>(a.tgt) + (long long)row * a.V * esz;
    } else {
        const int d = row - a.B * R;
        r.b = d / a.N;
        r.i = d % a.N;
        r.base = static_cast<const char*>(a.dft) + (long long)d * a.V * esz;
    }
    return r;
}

// Bitmap of the penalty set restricted to tokens [c0, c0 + 32 nwords).
__device__ __forceinline__ void build_penalty_bits(const VerifySampleArgs& a, int b, int i, long long c0,
                                                   int nwords, uint32_t* bits) {
    for (int w = threadIdx.x; w < nwords; w += blockDim.x) bits[w] = 0u;
    __syncthreads();
    const int total = a.H + i;
    for (int j = threadIdx.x; j < total; j += blockDim.x) {
        const int t = j < a.H ? a.hist[(long long)b * a.hist_stride + j]
                              : a.drafts[(long long)b * a.N + (j - a.H)];
        const long long rel = (long long)t - c0;
        if (t >= 0 && t < a.V && rel >= 0 && rel < (long long)nwords * 32) atomicOr(&bits[rel >> 5], 1u << (rel & 31));
    }
    __syncthreads();
}

__device__ __forceinline__ float row_value(const VerifySampleArgs& a, const void* base, long long x) {
    return a.bf16 ? bf16_to_f32(reinterpret_cast<const uint16_t*>(base)[x]) : reinterpret_cast<const float*>(base)[x];
}

__device__ __forceinline__ float key_to_float(uint32_t key) {
    const uint32_t u = (key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key;
    return __uint_as_float(u);
}

// Scan of one (row, chunk) item.  mode 0: fold the max scaled logit into
// rowmax[row]; mode 1: append every token with exp_cw(l - lmax) >= min_p to
// the row's candidate list.
static __device__ void sample_scan_item(const VerifySampleArgs& a, int row, long long c0, long long c1, int mode,
                                 uint32_t* bits, unsigned long long* red64) {
    const RowInfo ri = row_info(a, row);
    const int nwords = (int)((c1 - c0 + 31) / 32);
    build_penalty_bits(a, ri.b, ri.i, c0, nwords, bits);
    float lmax = 0.f, lthr = 0.f;
    if (mode == 1) {
        lmax = key_to_float((uint32_t)(__ldcg(a.rowmax + row) >> 32));
        // cheap superset test before the exact weight: exp_cw(d) >= min_p needs d >= ln(min_p) - tiny
        lthr = a.min_p > 0.f ? lmax + logf(a.min_p) - 1e-3f : -INFINITY;
    }
    unsigned long long best = 0ull;
    for (long long x = c0 + threadIdx.x; x < c1; x += blockDim.x) {
        const float z = row_value(a, ri.base, x);
        const long long rel = x - c0;
        const bool pen = (bits[rel >> 5] >> (rel & 31)) & 1u;
        const float l = scaled_logit(a, z, pen);
        if (mode == 0) {
            const unsigned long long k = pack_argmax(l, (uint32_t)x);
            best = k > best ? k : best;
        } else if (l >= lthr) {
            const float wx = exp_cw(__fsub_rn(l, lmax));
            if (wx >= a.min_p) {
                const unsigned int slot = atomicAdd(a.cand_cnt + row, 1u);
                if (slot < (unsigned)kCandCap) {
                    a.cand_id[(long long)row * kCandCap + slot] = (int32_t)x;
                    a.cand_w[(long long)row * kCandCap + slot] = wx;
                } else {
                    atomicCAS(&a.hdr->status, 0, MTP_ERR_CAPACITY);
                }
            }
        }
    }
    if (mode == 0) {
        best = warp_max_u64(best);
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        __syncthreads();
        if (lane == 0) red64[warp] = best;
        __syncthreads();
        if (threadIdx.x == 0) {
            unsigned long long m = 0ull;
            for (int w = 0; w < kWarps; ++w) m = red64[w] > m ? red64[w] : m;
            atomicMax(a.rowmax + row, m);
        }
    }
    __syncthreads();
}

// Sort one row's candidates by (w desc, id asc), cut by top-p, store ids /
// weights in order, n_keep and the kept mass.  Sums are sequential (thread 0).
static __device__ void sample_sort_row(const VerifySampleArgs& a, int row, unsigned long long* keys, float* wsh) {
    unsigned int n = __ldcg(a.cand_cnt + row);
    if (n > (unsigned)kCandCap) n = kCandCap;
    unsigned int P = 32;
    while (P < n) P <<= 1;
    for (unsigned int j = threadIdx.x; j < P; j += blockDim.x) {
        if (j < n) {
            const float w = __ldcg(a.cand_w + (long long)row * kCandCap + j);
            const int32_t id = __ldcg(a.cand_id + (long long)row * kCandCap + j);
            keys[j] = ((unsigned long long)(~ordered_key(w)) << 32) | (uint32_t)id;
        } else {
            keys[j] = ~0ull;
        }
    }
    __syncthreads();
    for (unsigned int k = 2; k <= P; k <<= 1) {
        for (unsigned int j = k >> 1; j > 0; j >>= 1) {
            for (unsigned int t = threadIdx.x; t < P; t += blockDim.x) {
                const unsigned int p2 = t ^ j;
                if (p2 > t) {
                    const bool up = (t & k) == 0;
                    const unsigned long long x = keys[t], y = keys[p2];
                    if ((x > y) == up) { keys[t] = y; keys[p2] = x; }
                }
            }
            __syncthreads();
        }
    }
    for (unsigned int j = threadIdx.x; j < n; j += blockDim.x) wsh[j] = key_to_float(~(uint32_t)(keys[j] >> 32));
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned int keep = n;
        if (a.top_p < 1.f) {
            float tot = 0.f;
            for (unsigned int j = 0; j < n; ++j) tot = __fadd_rn(tot, wsh[j]);
            float cum = 0.f;
            for (unsigned int j = 0; j < n; ++j) {
                cum = __fadd_rn(cum, wsh[j]);
                if (__fdiv_rn(cum, tot) >= a.top_p) { keep = j + 1; break; }
            }
        }
        float kept = 0.f;
        for (unsigned int j = 0; j < keep; ++j) kept = __fadd_rn(kept, wsh[j]);
        a.n_keep[row] = (int)keep;
        a.w_keep[row] = kept;
    }
    for (unsigned int j = threadIdx.x; j < n; j += blockDim.x) {
        a.cand_id[(long long)row * kCandCap + j] = (int32_t)(uint32_t)(keys[j] & 0xFFFFFFFFull);
        a.cand_w[(long long)row * kCandCap + j] = wsh[j];
    }
    __syncthreads();
}

// weight of token x in a sorted row (0 if not kept); warp-cooperative
__device__ __forceinline__ float row_weight(const VerifySampleArgs& a, int row, int32_t x) {
    const int n = __ldcg(a.n_keep + row);
    float w = 0.f;
    for (int j = threadIdx.x & 31; j < n; j += 32)
        if (__ldcg(a.cand_id + (long long)row * kCandCap + j) == x) w = __ldcg(a.cand_w + (long long)row * kCandCap + j);
    return warp_max(w);
}

// inverse-CDF pick: the first j with u * total < w_0 + ... + w_j, sums in order
template <class WF>
__device__ __forceinline__ int pick_index_seq(int n, float total, float u, WF wfn) {
    const float target = __fmul_rn(u, total);
    float acc = 0.f;
    for (int j = 0; j < n; ++j) {
        acc = __fadd_rn(acc, wfn(j));
        if (target < acc) return j;
    }
    return n > 0 ? n - 1 : 0;
}

// One warp walks sequence b's rows (lane 0 takes the decisions).
static __device__ void sample_decide(const VerifySampleArgs& a, int b) {
    const int lane = threadIdx.x & 31;
    const int R = a.N + 1;
    int32_t* out = a.out_tokens + (long long)b * R;
    int i = 0;
    for (; i < a.N; ++i) {
        const int trow = b * R + i;
        const int drow = a.B * R + b * a.N + i;
        const int32_t x = a.drafts[(long long)b * a.N + i];
        const float px = __fdiv_rn(row_weight(a, trow, x), __ldcg(a.w_keep + trow));
        const float qx = __fdiv_rn(row_weight(a, drow, x), __ldcg(a.w_keep + drow));
        const float u = philox_uniform(a.seed, a.offset, (uint32_t)b, (uint32_t)i, 1u);
        if (u < __fdiv_rn(px, qx)) {
            if (lane == 0) out[i] = x;
            continue;
        }
        // residual max(p - q, 0) over p's kept candidates, in p's order
        const int np = __ldcg(a.n_keep + trow);
        const float Wt = __ldcg(a.w_keep + trow), Wd = __ldcg(a.w_keep + drow);
        const long long tb = (long long)trow * kCandCap;
        float Rt = 0.f;
        for (int j = 0; j < np; ++j) {
            const float pj = __fdiv_rn(__ldcg(a.cand_w + tb + j), Wt);
            const float qj = __fdiv_rn(row_weight(a, drow, __ldcg(a.cand_id + tb + j)), Wd);
            const float r = pj > qj ? __fsub_rn(pj, qj) : 0.f;
            if (lane == 0) a.resid[(long long)b * kCandCap + j] = r;
            Rt = __fadd_rn(Rt, r);
        }
        __syncwarp();
        const float u2 = philox_uniform(a.seed, a.offset, (uint32_t)b, (uint32_t)i, 2u);
        int j;
        if (Rt > 0.f) j = pick_index_seq(np, Rt, u2, [&](int jj) { return __ldcg(a.resid + (long long)b * kCandCap + jj); });
        else j = pick_index_seq(np, Wt, u2, [&](int jj) { return __ldcg(a.cand_w + tb + jj); });
        if (lane == 0) out[i] = __ldcg(a.cand_id + tb + j);
        break;
    }
    if (i == a.N) {
        const int trow = b * R + a.N;
        const long long tb = (long long)trow * kCandCap;
        const float u3 = philox_uniform(a.seed, a.offset, (uint32_t)b, (uint32_t)a.N, 3u);
        const int j = pick_index_seq(__ldcg(a.n_keep + trow), __ldcg(a.w_keep + trow), u3,
                                     [&](int jj) { return __ldcg(a.cand_w + tb + jj); });
        if (lane == 0) out[a.N] = __ldcg(a.cand_id + tb + j);
    }
    if (lane == 0) {
        for (int j = i + 1; j < R; ++j) out[j] = -1;
        a.out_n_accept[b] = i;
    }
}

// Draft sampling: one warp draws sequence b's token at step a.draft_k from
// its sorted row with the uniform of (b, draft_k, purpose 0).
__device__ __forceinline__ int32_t sample_pick_draft(const VerifySampleArgs& a, int b) {
    const long long tb = (long long)b * kCandCap;
    const float u = philox_uniform(a.seed, a.offset, (uint32_t)b, (uint32_t)a.draft_k, 0u);
    const int j = pick_index_seq(__ldcg(a.n_keep + b), __ldcg(a.w_keep + b), u,
                                 [&](int jj) { return __ldcg(a.cand_w + tb + jj); });
    return __ldcg(a.cand_id + tb + j);
}

}  // namespace mtp
