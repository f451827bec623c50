// verify.cu -- verify-accept kernels.
//
// Greedy ("MTP decoding (--mtp)", How it is wired): one launch.  The (1+N)
// rows of every sequence are split into V-chunks; each CTA reduces its chunk
// to a packed (value, index) key and folds it into the row's slot with one
// 64-bit atomicMax, so the result does not depend on CTA order.  The last CTA
// to finish (a counter in the workspace header) turns the row argmaxes into
// the accepted prefix and the bonus token.
//
// Exact sampling ("opus-mtp-turbo: Track 1 report", item 4): one cooperative
// launch with four phases separated by grid barriers:
//   1. penalised row maxima           (all rows, V split across CTAs)
//   2. min-p candidate collection     (all rows, V split across CTAs)
//   3. sort by (p desc, id asc), top-p cut   (one CTA per row)
//   4. accept / residual / bonus walk        (one warp per sequence)
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "verify.cuh"

namespace mtp {

// ---------------------------------------------------------------------------
// greedy
// ---------------------------------------------------------------------------

template <typename T>
__device__ __forceinline__ void chunk_argmax(const T* row, long long c0, long long c1,
                                             unsigned long long& best);

template <>
__device__ __forceinline__ void chunk_argmax<uint16_t>(const uint16_t* row, long long c0, long long c1,
                                                       unsigned long long& best) {
    // scalar head up to a 16-byte boundary, 8-wide body, scalar tail
    long long a = c0;
    while (a < c1 && ((reinterpret_cast<uintptr_t>(row + a) & 15) != 0)) {
        if (((a - c0) % blockDim.x) == threadIdx.x) {
            unsigned long long k = pack_argmax(bf16_to_f32(row[a]), (uint32_t)a);
            best = k > best ? k : best;
        }
        ++a;
    }
    const long long nvec = (c1 - a) / 8;
    const uint4* v = reinterpret_cast<const uint4*>(row + a);
    for (long long i = threadIdx.x; i < nvec; i += blockDim.x) {
        uint4 w = ld_stream16(v + i);
        const uint32_t base = (uint32_t)(a + i * 8);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            unsigned long long k0 = pack_argmax(bf16_lo(ws[j]), base + 2 * j);
            unsigned long long k1 = pack_argmax(bf16_hi(ws[j]), base + 2 * j + 1);
            best = k0 > best ? k0 : best;
            best = k1 > best ? k1 : best;
        }
    }
    for (long long t = a + nvec * 8 + threadIdx.x; t < c1; t += blockDim.x) {
        unsigned long long k = pack_argmax(bf16_to_f32(row[t]), (uint32_t)t);
        best = k > best ? k : best;
    }
}

template <>
__device__ __forceinline__ void chunk_argmax<float>(const float* row, long long c0, long long c1,
                                                    unsigned long long& best) {
    long long a = c0;
    while (a < c1 && ((reinterpret_cast<uintptr_t>(row + a) & 15) != 0)) {
        if (((a - c0) % blockDim.x) == threadIdx.x) {
            unsigned long long k = pack_argmax(row[a], (uint32_t)a);
            best = k > best ? k : best;
        }
        ++a;
    }
    const long long nvec = (c1 - a) / 4;
    const uint4* v = reinterpret_cast<const uint4*>(row + a);
    for (long long i = threadIdx.x; i < nvec; i += blockDim.x) {
        uint4 w = ld_stream16(v + i);
        const uint32_t base = (uint32_t)(a + i * 4);
        unsigned long long k;
        k = pack_argmax(__uint_as_float(w.x), base + 0); best = k > best ? k : best;
        k = pack_argmax(__uint_as_float(w.y), base + 1); best = k > best ? k : best;
        k = pack_argmax(__uint_as_float(w.z), base + 2); best = k > best ? k : best;
        k = pack_argmax(__uint_as_float(w.w), base + 3); best = k > best ? k : best;
    }
    for (long long t = a + nvec * 4 + threadIdx.x; t < c1; t += blockDim.x) {
        unsigned long long k2 = pack_argmax(row[t], (uint32_t)t);
        best = k2 > best ? k2 : best;
    }
}

template <typename T>
__global__ void __launch_bounds__(256) verify_greedy_kernel(VerifyGreedyArgs a) {
    const int row = blockIdx.y;                  // b * (1+N) + i
    const long long V = a.V;
    const long long chunk = (V + gridDim.x - 1) / gridDim.x;
    const long long c0 = (long long)blockIdx.x * chunk;
    const long long c1 = c0 + chunk < V ? c0 + chunk : V;
    const T* rowp = reinterpret_cast<const T*>(a.logits) + (long long)row * V;

    unsigned long long best = 0ull;
    if (c0 < c1) chunk_argmax<T>(rowp, c0, c1, best);
    best = warp_max_u64(best);
    __shared__ unsigned long long sbest[8];
    __shared__ int s_last;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) sbest[warp] = best;
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned long long m = 0ull;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) m = sbest[w] > m ? sbest[w] : m;
        if (c0 < c1) atomicMax(a.amax + row, m);
        __threadfence();
        const unsigned int total = gridDim.x * gridDim.y;
        s_last = (atomicAdd(&a.hdr->done, 1u) == total - 1u);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    // last CTA: longest matching prefix + bonus for every sequence
    const int R = a.N + 1;
    for (int b = threadIdx.x; b < a.B; b += blockDim.x) {
        int k = 0;
        int32_t* out = a.out_tokens + (long long)b * R;
        for (;;) {
            const unsigned long long m = __ldcg(a.amax + (long long)b * R + k);
            const int32_t t = (int32_t)unpack_index(m);
            if (k < a.N && a.drafts[(long long)b * a.N + k] == t) { out[k] = t; ++k; continue; }
            out[k] = t;
            break;
        }
        for (int j = k + 1; j < R; ++j) out[j] = -1;
        a.out_n_accept[b] = k;
    }
}

cudaError_t launch_verify_greedy(const VerifyGreedyArgs& a, int ldtype, int num_sms, cudaStream_t s) {
    const long long rows = (long long)a.B * (a.N + 1);
    long long split = (4LL * num_sms + rows - 1) / rows;
    const long long max_split = (a.V + 2047) / 2048;
    if (split > max_split) split = max_split;
    if (split < 1) split = 1;
    dim3 grid((unsigned)split, (unsigned)rows);
    if (ldtype == MTP_DTYPE_BF16)
        verify_greedy_kernel<uint16_t><<<grid, 256, 0, s>>>(a);
    else
        verify_greedy_kernel<float><<<grid, 256, 0, s>>>(a);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// exact sampling
// ---------------------------------------------------------------------------

// penalised logit (before temperature) of token x with raw value z
__device__ __forceinline__ float penalise(float z, float rep, float pres) {
    float y = z > 0.f ? z / rep : z * rep;
    return y - pres;
}

// Row geometry: rows [0, B(1+N)) are target rows (b, i), rows [B(1+N),
// B(1+N) + B N) are draft rows (b, i).  Penalty set of (b, i): hist[b][*] u
// drafts[b][0..i-1].
struct RowInfo {
    const void* base;  // first element of the row
    int b, i;
};

__device__ __forceinline__ RowInfo row_info(const VerifySampleArgs& a, int row) {
    RowInfo r;
    const int R = a.N + 1;
    const long long esz = a.bf16 ? 2 : 4;
    if (row < a.B * R) {
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

// Build a bitmap of the penalty set restricted to tokens [c0, c0 + nbits) in
// shared memory (nbits rounded up to a multiple of 32).
__device__ void build_penalty_bits(const VerifySampleArgs& a, int b, int i, long long c0, int nwords,
                                   uint32_t* bits) {
    for (int w = threadIdx.x; w < nwords; w += blockDim.x) bits[w] = 0u;
    __syncthreads();
    const int total = a.H + i;
    for (int j = threadIdx.x; j < total; j += blockDim.x) {
        const int t = j < a.H ? a.hist[(long long)b * a.H + j] : a.drafts[(long long)b * a.N + (j - a.H)];
        const long long rel = (long long)t - c0;
        if (t >= 0 && t < a.V && rel >= 0 && rel < (long long)nwords * 32)
            atomicOr(&bits[rel >> 5], 1u << (rel & 31));
    }
    __syncthreads();
}

__device__ __forceinline__ float row_value(const VerifySampleArgs& a, const void* base, long long x) {
    return a.bf16 ? bf16_to_f32(reinterpret_cast<const uint16_t*>(base)[x])
                  : reinterpret_cast<const float*>(base)[x];
}

// penalised, temperature-scaled logit of token x (bitmap lookup)
__device__ __forceinline__ float scaled_logit(const VerifySampleArgs& a, float z, bool pen) {
    const float y = pen ? penalise(z, a.rep, a.pres) : z;
    return y / a.temp;
}

// Phase 1 / 2 body over one (row, chunk) item.  mode 0: fold the max of the
// scaled logits into rowmax[row]; mode 1: append every token with
// exp(l - lmax) >= min_p to the row's candidate list.
__device__ void sample_scan_item(const VerifySampleArgs& a, int row, long long c0, long long c1, int mode,
                                 uint32_t* bits, unsigned long long* red64) {
    const RowInfo ri = row_info(a, row);
    const int nwords = (int)((c1 - c0 + 31) / 32);
    build_penalty_bits(a, ri.b, ri.i, c0, nwords, bits);
    float lmax = 0.f;
    if (mode == 1) {
        const unsigned long long m = __ldcg(a.rowmax + row);
        // the max was folded as a packed key of the scaled logit; recover the value
        const uint32_t key = (uint32_t)(m >> 32);
        const uint32_t u = (key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key;
        lmax = __uint_as_float(u);
    }
    const float lthr = mode == 1 ? lmax + __logf(a.min_p > 0.f ? a.min_p : 1e-30f) - 1e-3f : 0.f;
    unsigned long long best = 0ull;
    for (long long x = c0 + threadIdx.x; x < c1; x += blockDim.x) {
        const float z = row_value(a, ri.base, x);
        const long long rel = x - c0;
        const bool pen = (bits[rel >> 5] >> (rel & 31)) & 1u;
        const float l = scaled_logit(a, z, pen);
        if (mode == 0) {
            const unsigned long long k = pack_argmax(l, (uint32_t)x);
            best = k > best ? k : best;
        } else if (l >= lthr || a.min_p <= 0.f) {
            const float w = __expf(l - lmax);
            const float wx = expf(l - lmax);
            (void)w;
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

// Phase 3: sort one row's candidates by (w desc, id asc), cut by top-p and
// store ids / weights in order plus n_keep and the kept mass.
__device__ void sample_sort_row(const VerifySampleArgs& a, int row, unsigned long long* keys, float* wsh) {
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
    // bitonic sort, ascending keys = weight descending, id ascending
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
    // weights in sorted order, then a sequential-order prefix scan by warp 0
    for (unsigned int j = threadIdx.x; j < n; j += blockDim.x) {
        const uint32_t key = ~(uint32_t)(keys[j] >> 32);
        const uint32_t u = (key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key;
        wsh[j] = __uint_as_float(u);
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        // total mass of the min-p set
        float tot = 0.f;
        for (unsigned int base = 0; base < n; base += 32) {
            float v = base + lane < n ? wsh[base + lane] : 0.f;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                float t = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += t;
            }
            tot += __shfl_sync(0xffffffffu, v, 31);
        }
        // first j whose share of the mass reaches top_p
        unsigned int keep = n;
        if (a.top_p < 1.f) {
            float carry = 0.f;
            for (unsigned int base = 0; base < n && keep == n; base += 32) {
                float v = base + lane < n ? wsh[base + lane] : 0.f;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    float t = __shfl_up_sync(0xffffffffu, v, o);
                    if (lane >= o) v += t;
                }
                const float cum = carry + v;
                const bool hit = (base + lane < n) && (cum / tot >= a.top_p);
                const unsigned int mask = __ballot_sync(0xffffffffu, hit);
                if (mask) keep = base + __ffs(mask);
                carry += __shfl_sync(0xffffffffu, v, 31);
            }
        }
        // kept mass in order
        float kept = 0.f;
        for (unsigned int base = 0; base < keep; base += 32) {
            float v = base + lane < keep ? wsh[base + lane] : 0.f;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                float t = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += t;
            }
            kept += __shfl_sync(0xffffffffu, v, 31);
        }
        if (lane == 0) {
            a.n_keep[row] = (int)keep;
            a.w_keep[row] = kept;
        }
    }
    for (unsigned int j = threadIdx.x; j < n; j += blockDim.x) {
        a.cand_id[(long long)row * kCandCap + j] = (int32_t)(uint32_t)(keys[j] & 0xFFFFFFFFull);
        a.cand_w[(long long)row * kCandCap + j] = wsh[j];
    }
    __syncthreads();
}

// probability of token x under a sorted row (0 if not kept); warp-cooperative
__device__ __forceinline__ float row_prob(const VerifySampleArgs& a, int row, int32_t x) {
    const int n = __ldcg(a.n_keep + row);
    float w = 0.f;
    for (int j = threadIdx.x & 31; j < n; j += 32)
        if (__ldcg(a.cand_id + (long long)row * kCandCap + j) == x) w = __ldcg(a.cand_w + (long long)row * kCandCap + j);
    w = warp_max(w);
    return w / __ldcg(a.w_keep + row);
}

// inverse-CDF pick over weights wfn(j), j < n, walked in order: the first j
// with u * total < w_0 + ... + w_j.  Warp-cooperative; returns the index j.
template <class WF>
__device__ __forceinline__ int pick_index(int n, float total, float u, WF wfn) {
    const int lane = threadIdx.x & 31;
    const float target = u * total;
    float carry = 0.f;
    for (int base = 0; base < n; base += 32) {
        float v = base + lane < n ? wfn(base + lane) : 0.f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            float t = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += t;
        }
        const bool hit = (base + lane < n) && (target < carry + v);
        const unsigned int mask = __ballot_sync(0xffffffffu, hit);
        if (mask) return base + __ffs(mask) - 1;
        carry += __shfl_sync(0xffffffffu, v, 31);
    }
    return n > 0 ? n - 1 : 0;
}

// Phase 4: one warp walks sequence b's rows.
__device__ void sample_decide(const VerifySampleArgs& a, int b) {
    const int lane = threadIdx.x & 31;
    const int R = a.N + 1;
    int32_t* out = a.out_tokens + (long long)b * R;
    int i = 0;
    for (; i < a.N; ++i) {
        const int trow = b * R + i;
        const int drow = a.B * R + b * a.N + i;
        const int32_t x = a.drafts[(long long)b * a.N + i];
        const float px = row_prob(a, trow, x);
        const float qx = row_prob(a, drow, x);
        const float u = philox_uniform(a.seed, a.offset, (uint32_t)b, (uint32_t)i, 1u);
        if (u < px / qx) {
            if (lane == 0) out[i] = x;
            continue;
        }
        // residual max(p - q, 0) over p's kept candidates, in p's order
        const int np = __ldcg(a.n_keep + trow);
        const float Wt = __ldcg(a.w_keep + trow);
        const long long tb = (long long)trow * kCandCap;
        // q of each of p's candidates: a warp-wide search per candidate
        float R_tot = 0.f;
        for (int j = 0; j < np; ++j) {
            const float pj = __ldcg(a.cand_w + tb + j) / Wt;
            const float qj = row_prob(a, drow, __ldcg(a.cand_id + tb + j));
            const float r = pj > qj ? pj - qj : 0.f;
            if (lane == 0) a.resid[(long long)b * kCandCap + j] = r;
            R_tot += r;
        }
        __syncwarp();
        const float u2 = philox_uniform(a.seed, a.offset, (uint32_t)b, (uint32_t)i, 2u);
        int j;
        if (R_tot > 0.f) {
            j = pick_index(np, R_tot, u2, [&](int jj) { return __ldcg(a.resid + (long long)b * kCandCap + jj); });
        } else {
            j = pick_index(np, Wt, u2, [&](int jj) { return __ldcg(a.cand_w + tb + jj); });
        }
        if (lane == 0) out[i] = __ldcg(a.cand_id + tb + j);
        break;
    }
    if (i == a.N) {
        const int trow = b * R + a.N;
        const long long tb = (long long)trow * kCandCap;
        const float u3 = philox_uniform(a.seed, a.offset, (uint32_t)b, (uint32_t)a.N, 3u);
        const int j = pick_index(__ldcg(a.n_keep + trow), __ldcg(a.w_keep + trow), u3,
                                 [&](int jj) { return __ldcg(a.cand_w + tb + jj); });
        if (lane == 0) out[a.N] = __ldcg(a.cand_id + tb + j);
    }
    if (lane == 0) {
        for (int j = i + 1; j < R; ++j) out[j] = -1;
        a.out_n_accept[b] = i;
    }
}

__global__ void __launch_bounds__(kThreads, 1) verify_sample_kernel(VerifySampleArgs a) {
    extern __shared__ __align__(16) unsigned char smem[];
    unsigned int epoch = 0;
    const int rows = a.B * (a.N + 1) + a.B * a.N;
    const long long chunks = (a.V + kScanChunk - 1) / kScanChunk;
    const long long items = (long long)rows * chunks;
    uint32_t* bits = reinterpret_cast<uint32_t*>(smem);
    unsigned long long* red64 = reinterpret_cast<unsigned long long*>(smem + kScanChunk / 8);
    for (int mode = 0; mode < 2; ++mode) {
        for (long long it = blockIdx.x; it < items; it += gridDim.x) {
            const int row = (int)(it / chunks);
            const long long c0 = (it % chunks) * kScanChunk;
            const long long c1 = c0 + kScanChunk < a.V ? c0 + kScanChunk : a.V;
            sample_scan_item(a, row, c0, c1, mode, bits, red64);
        }
        if (!grid_barrier(a.hdr, epoch, a.timeout_ns, gridDim.x)) return;
    }
    unsigned long long* keys = reinterpret_cast<unsigned long long*>(smem);
    float* wsh = reinterpret_cast<float*>(smem + kCandCap * sizeof(unsigned long long));
    for (int row = blockIdx.x; row < rows; row += gridDim.x) sample_sort_row(a, row, keys, wsh);
    if (!grid_barrier(a.hdr, epoch, a.timeout_ns, gridDim.x)) return;
    const int gw = blockIdx.x * kWarps + (threadIdx.x >> 5);
    for (int b = gw; b < a.B; b += gridDim.x * kWarps) sample_decide(a, b);
}

size_t verify_sample_smem_bytes() {
    const size_t scan = kScanChunk / 8 + kWarps * sizeof(unsigned long long);
    const size_t sort = kCandCap * (sizeof(unsigned long long) + sizeof(float));
    return scan > sort ? scan : sort;
}

cudaError_t launch_verify_sample(const VerifySampleArgs& a, int grid, cudaStream_t s) {
    const size_t smem = verify_sample_smem_bytes();
    cudaError_t e = cudaFuncSetAttribute(verify_sample_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    VerifySampleArgs copy = a;
    void* args[] = {&copy};
    return cudaLaunchCooperativeKernel((const void*)verify_sample_kernel, dim3(grid), dim3(kThreads), args, smem, s);
}

int verify_sample_max_grid(int num_sms) {
    int per_sm = 0;
    const size_t smem = verify_sample_smem_bytes();
    cudaFuncSetAttribute(verify_sample_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, verify_sample_kernel, kThreads, smem) != cudaSuccess)
        return 0;
    return per_sm * num_sms;
}

}  // namespace mtp
