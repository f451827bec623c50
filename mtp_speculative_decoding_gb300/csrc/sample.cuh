// sample.cuh -- sample_dist and exact speculative acceptance on the GPU
// ("opus-mtp-turbo: Track 1 report", item 4: penalties over history + window
// inputs, temperature, min-p, top-p; accept with p(x)/q(x), on rejection a
// draw from norm(max(p - q, 0)), a fully accepted window draws its bonus from
// the last target row).
//
// The sampler's arithmetic decides integers, so every step that feeds a
// decision is IEEE fp32 with its rounding written out (no contraction):
// penalised logit z / r or z * r, minus the presence penalty, divided by the
// temperature; the difference l - lmax; the weight w = exp(l - lmax) rounded
// once to fp32 (the exponential is evaluated in fp64); every sum runs
// sequentially in (w desc, id asc) order.
//
// One pass over the logits.  A row (one sequence's target or draft logits of
// one window position) is cut into pieces; a CTA streams a piece with 16-byte
// loads, keeps the running maximum of the raw logits, and keeps every token
// that can still reach the min-p cut against that running maximum -- a
// superset of the final candidates, since the maximum only grows.  The
// penalty set (at most H + N tokens) is left out of the piece's survivors
// and evaluated exactly by the row's finishing CTA; a piece whose maximum
// belongs only to penalised tokens sends its row to an exact rescan.  The
// last piece of a row to finish (a counter) takes the row's maximum, applies
// the exact min-p rule, sorts, cuts by top-p and stores the kept set; the
// last row of a sequence to finish walks the sequence's accept / residual /
// bonus decisions.  No grid-wide barrier: a plain launch suffices.  If a
// buffer overflows, the row's finishing CTA rescans the row, so the result
// stays exact.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "common.cuh"

namespace mtp {

constexpr int kCandCap = 4096;     // largest kept (min-p) set of one row
constexpr int kPieceMax = 65536;   // tokens per piece at most
constexpr int kPieceBuf = 4096;    // survivors a piece may hold in shared memory
constexpr int kRowBufCap = 8192;   // survivors a row may hold in its buffer

// dynamic shared memory of sample_piece: the row's penalty list (or, in a
// rescan, a window's penalty bitmap plus a spare word), then a region for the
// piece's survivors or the finishing CTA's sort keys (8 bytes each), then the
// finishing CTA's fp32 weights
constexpr int kPenMax = 1024;      // penalty-list entries (H + window position) kept in shared memory
constexpr int kBloomWords = 64;    // a 2048-bit filter over the penalty list (bit = id mod 2048)
constexpr size_t kSampBitmapBytes = (kPieceMax / 32 + 4) * 4;
static_assert(kSampBitmapBytes >= (size_t)(kPenMax + kBloomWords) * 4 + 16, "penalty list fits the bitmap area");
constexpr int kRankSortMax = 512;  // kept sets up to this size are sorted by rank (one pass), larger by bitonic
constexpr size_t kSampKeyBytes = (size_t)kCandCap * 8 > (size_t)kPieceBuf * 8 ? (size_t)kCandCap * 8 : (size_t)kPieceBuf * 8;
constexpr size_t kSampleSmem = kSampBitmapBytes + kSampKeyBytes + (size_t)kCandCap * 4;

// What a sampling launch works on.
//   mode 0 (verify): rows [0, B(1+N)) are target rows (b, i), rows
//     [B(1+N), B(1+N) + B N) draft rows (b, i); penalty set hist[b] u
//     drafts[b][0..i-1]; the last row of a sequence walks its decisions.
//   mode 1 (draw): row b is sequence b's logits at window position draw_i
//     (base0 + b * draw_ld); penalty set hist[b] u drafts[b][0..draw_i-1];
//     the row's finishing CTA draws the token with the uniform of
//     (b, draw_i, purpose 0) and writes it to out_draw[b * out_draw_ld +
//     draw_i] and/or out_amax[b] (as a packed key).
struct SampleJob {
    const void* base0;   // mode 0: target [B, 1+N, V]; mode 1: first row
    const void* base1;   // mode 0: draft [B, N, V]
    int f32;             // element type: 1 fp32, 0 bf16
    int mode;
    int B, N;
    long long V;
    long long draw_ld;   // mode 1: elements from row b to row b + 1
    int draw_i;
    const int32_t* drafts;   // penalty source and (mode 0) the drafted tokens, [B][drafts_ld]
    int drafts_ld;
    const int32_t* hist;     // [B][hist_ld], H used
    int H, hist_ld;
    float temp, top_p, min_p, rep, pres;
    unsigned long long seed, offset;
    int32_t* out_tokens;     // mode 0: [B, 1+N]
    int32_t* out_n_accept;   // mode 0: [B]
    int32_t* out_draw;       // mode 1 (or null)
    int out_draw_ld;
    unsigned long long* out_amax;   // mode 1 (or null): packed key of the drawn token
    WsHeader* hdr;
    // per-row state (zero before first use; every finishing CTA re-zeroes its row)
    unsigned int* row_max;    // ordered key of the row's largest scaled logit
    unsigned int* row_cnt;    // survivors in row_buf
    unsigned int* row_ovf;    // a piece or the row buffer overflowed
    unsigned int* row_done;   // pieces finished
    unsigned int* seq_done;   // mode 0: rows finished per sequence
    int2* row_buf;            // [rows][rcap] (id, scaled logit bits)
    int rcap;
    int32_t* keep_id;         // mode 0: [rows][ccap] kept ids in (w desc, id asc) order
    float* keep_w;            // mode 0: their weights
    int ccap;
    int32_t* n_keep;          // mode 0: [rows]
    float* w_keep;            // mode 0: [rows] kept weight sums
    int piece_len;            // tokens per piece (multiple of 32, <= kPieceMax)
    int ppr;                  // pieces per row
    unsigned int* next_piece; // standalone launches: pieces handed out so far past the first grid (zeroed)
};

__host__ __device__ inline int sample_rows(const SampleJob& j) {
    return j.mode == 0 ? j.B * (j.N + 1) + j.B * j.N : j.B;
}

// scaled logit of a penalised token: z > 0: z / r, else z * r; minus pres; / temp
__device__ __forceinline__ float penalised_logit(const SampleJob& j, float z) {
    float y = z > 0.f ? __fdiv_rn(z, j.rep) : __fmul_rn(z, j.rep);
    y = __fsub_rn(y, j.pres);
    return __fdiv_rn(y, j.temp);
}

// candidate weight: exp(l - M) with the difference in fp32 and the
// exponential in fp64, rounded once to fp32
__device__ __forceinline__ float cand_weight(float l, float M) {
    const float d = __fsub_rn(l, M);
    return __double2float_rn(exp((double)d));
}

__device__ __forceinline__ float key_to_float(uint32_t key) {
    const uint32_t u = (key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key;
    return __uint_as_float(u);
}
// a maximum kept as an ordered key; 0 (nothing folded yet) reads as -inf
__device__ __forceinline__ float key_max(uint32_t key) { return key ? key_to_float(key) : -INFINITY; }
__device__ __forceinline__ float shared_max(const unsigned int* k) {
    return key_max(*reinterpret_cast<const volatile unsigned int*>(k));
}

struct RowRef {
    const void* base;   // row start
    int b, i;           // sequence, window position
};

__device__ __forceinline__ RowRef row_ref(const SampleJob& j, int row) {
    RowRef r;
    const long long esz = j.f32 ? 4 : 2;
    if (j.mode == 1) {
        r.b = row;
        r.i = j.draw_i;
        r.base = static_cast<const char*>(j.base0) + (long long)row * j.draw_ld * esz;
        return r;
    }
    const int R = j.N + 1;
    if (row < j.B * R) {
        r.b = row / R;
        r.i = row % R;
        r.base = static_cast<const char*>(j.base0) + (long long)row * j.V * esz;
    } else {
        const int d = row - j.B * R;
        r.b = d / j.N;
        r.i = d % j.N;
        r.base = static_cast<const char*>(j.base1) + (long long)d * j.V * esz;
    }
    return r;
}

// Loads of logits go through L2 (.cg): the draft kernel samples logits it
// wrote itself earlier in the same launch, which rules out the read-only path.
__device__ __forceinline__ float row_elem(const SampleJob& j, const void* base, long long x) {
    return j.f32 ? __ldcg(reinterpret_cast<const float*>(base) + x)
                 : bf16_to_f32(__ldcg(reinterpret_cast<const uint16_t*>(base) + x));
}

// Penalty bitmap of tokens [c0, c0 + 32 nwords) for (b, i); words past the
// range stay zero.  Whole CTA.
__device__ __forceinline__ void build_bitmap(const SampleJob& j, int b, int i, long long c0, int nwords,
                                             uint32_t* bits) {
    for (int w = threadIdx.x; w < nwords + 1; w += blockDim.x) bits[w] = 0u;
    __syncthreads();
    const int total = j.H + i;
    for (int t = threadIdx.x; t < total; t += blockDim.x) {
        const int x = t < j.H ? j.hist[(long long)b * j.hist_ld + t] : j.drafts[(long long)b * j.drafts_ld + (t - j.H)];
        const long long rel = (long long)x - c0;
        if (x >= 0 && x < j.V && rel >= 0 && rel < (long long)nwords * 32) atomicOr(&bits[rel >> 5], 1u << (rel & 31));
    }
    __syncthreads();
}

// 8 penalty bits starting at relative token rel (may straddle two words)
__device__ __forceinline__ uint32_t pen_bits8(const uint32_t* bits, long long rel) {
    const int w = (int)(rel >> 5), o = (int)(rel & 31);
    uint32_t v = bits[w] >> o;
    if (o > 24) v |= bits[w + 1] << (32 - o);
    return v & 0xFFu;
}

// ln(min_p) as the survivors' threshold offset (-inf when min_p == 0)
__device__ __forceinline__ float log_min_p(const SampleJob& j) { return j.min_p > 0.f ? logf(j.min_p) : -INFINITY; }

// the survivors' threshold below a maximum m (in the units of m), with a
// relative slack that covers every rounding between here and the exact rule
__device__ __forceinline__ float survive_thr(float m, float off) {
    if (!(off > -INFINITY) || !(m > -INFINITY)) return -INFINITY;
    const float t = m + off;
    return t - 1e-3f * (fabsf(m) + fabsf(off)) - 1e-30f;
}

// ---------------------------------------------------------------------------
// one piece: stream, keep survivors, hand them to the row
// ---------------------------------------------------------------------------

// Appends (x, l) to the piece buffer.
__device__ __forceinline__ void piece_push(unsigned int* cnt, int2* buf, long long x, float l) {
    const unsigned int s = atomicAdd(cnt, 1u);
    if (s < (unsigned)kPieceBuf) buf[s] = make_int2((int)x, __float_as_int(l));
}

// largest of the 16 bytes' values (NaN ignored), bf16 pairs compared packed
__device__ __forceinline__ float vec_max(const uint4& w, uint16_t) {
    const __nv_bfloat162 a = __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&w.x), *reinterpret_cast<const __nv_bfloat162*>(&w.y));
    const __nv_bfloat162 c = __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&w.z), *reinterpret_cast<const __nv_bfloat162*>(&w.w));
    const __nv_bfloat162 m = __hmax2(a, c);
    return fmaxf(__low2float(m), __high2float(m));
}
__device__ __forceinline__ float vec_max(const uint4& w, float) {
    return fmaxf(fmaxf(__uint_as_float(w.x), __uint_as_float(w.y)), fmaxf(__uint_as_float(w.z), __uint_as_float(w.w)));
}

// Streams tokens [c0, c1) of a row, folding their raw maximum into *zmax
// (ordered key) and keeping every token within the survivors' threshold of
// the running maximum (raw values; the penalty set is sorted out at the
// piece's end).  U vectors of 16 bytes in flight per thread.
template <typename T>
__device__ __forceinline__ void piece_stream(const SampleJob& j, const T* row, long long c0, long long c1,
                                             unsigned int* zmax, unsigned int* cnt, int2* buf) {
    constexpr int EPV = 16 / (int)sizeof(T);   // elements per vector
    constexpr int U = 8;
    const int lane = threadIdx.x & 31;
    const float off_z = j.temp * log_min_p(j);   // ln(min_p) in raw-logit units
    // unaligned head, then whole vectors, then the tail
    long long a = c0;
    while (a < c1 && (reinterpret_cast<uintptr_t>(row + a) & 15) != 0) ++a;
    const long long nvec = (c1 - a) / EPV;
    const long long tail0 = a + nvec * EPV;
    // head and tail elements: one per thread, before the vectors
    {
        float v = -INFINITY;
        long long xs = -1;
        const long long nh = a - c0, nt = c1 - tail0;
        if ((long long)threadIdx.x < nh) xs = c0 + threadIdx.x;
        else if ((long long)threadIdx.x < nh + nt) xs = tail0 + (threadIdx.x - nh);
        if (xs >= 0) v = row_elem(j, row, xs);
        const float m = warp_max(v);
        if (lane == 0 && m > -INFINITY) atomicMax(zmax, ordered_key(m));
        __syncwarp();
        const float run = fmaxf(m, shared_max(zmax));
        if (xs >= 0 && v >= survive_thr(run, off_z)) piece_push(cnt, buf, xs, v);
    }
    float run = shared_max(zmax);
    const uint4* vp = reinterpret_cast<const uint4*>(row + a);
    const long long step = (long long)blockDim.x * U;
    for (long long vb = 0; vb < nvec; vb += step) {   // the same trip count on every thread (shuffles below)
        const long long v0 = vb + threadIdx.x;
        uint4 w[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const long long v = v0 + (long long)u * blockDim.x;
            w[u] = v < nvec ? __ldcg(vp + v) : make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
        }
        float vm[U];
        float m = -INFINITY;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const long long v = v0 + (long long)u * blockDim.x;
            vm[u] = v < nvec ? vec_max(w[u], T()) : -INFINITY;
            m = fmaxf(m, vm[u]);
        }
        m = warp_max(m);
        if (lane == 0 && m > run) atomicMax(zmax, ordered_key(m));
        run = fmaxf(run, fmaxf(m, shared_max(zmax)));
        const float thr = survive_thr(run, off_z);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (vm[u] >= thr) {   // rare: some element of the vector survives
                const uint32_t ws[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
#pragma unroll
                for (int e = 0; e < EPV; ++e) {
                    const float z = sizeof(T) == 2 ? ((e & 1) ? bf16_hi(ws[e >> 1]) : bf16_lo(ws[e >> 1]))
                                                   : __uint_as_float(ws[e]);
                    if (z >= thr) piece_push(cnt, buf, a + (v0 + (long long)u * blockDim.x) * EPV + e, z);
                }
            }
        }
    }
}

// Loads (b, i)'s penalty list -- hist[b] then drafts[b][0..i-1], duplicates
// and out-of-range ids included -- into pen, and a 2048-bit filter of it
// after the list's kPenMax slots; returns the list's length, or -1 when it
// does not fit (kPenMax).  Whole CTA; synchronises.
__device__ __forceinline__ int load_penalty_list(const SampleJob& j, int b, int i, int32_t* pen) {
    const int total = j.H + i;
    if (total > kPenMax) return -1;
    uint32_t* bloom = reinterpret_cast<uint32_t*>(pen + kPenMax);
    for (int t = threadIdx.x; t < kBloomWords; t += blockDim.x) bloom[t] = 0u;
    __syncthreads();
    for (int t = threadIdx.x; t < total; t += blockDim.x) {
        const int x = t < j.H ? j.hist[(long long)b * j.hist_ld + t] : j.drafts[(long long)b * j.drafts_ld + (t - j.H)];
        pen[t] = x;
        atomicOr(&bloom[(x >> 5) & (kBloomWords - 1)], 1u << (x & 31));
    }
    __syncthreads();
    return total;
}

__device__ __forceinline__ bool in_list(const int32_t* pen, int n, int x) {
    const uint32_t* bloom = reinterpret_cast<const uint32_t*>(pen + kPenMax);
    if (!((bloom[(x >> 5) & (kBloomWords - 1)] >> (x & 31)) & 1u)) return false;
    bool f = false;
    for (int t = 0; t < n; ++t) f |= pen[t] == x;
    return f;
}

// the row's finishing work (defined below)
static __device__ void sample_finish_row(const SampleJob& j, int row, unsigned char* smem);

// L2 prefetch of piece `piece`'s bytes (one thread)
__device__ __forceinline__ void prefetch_piece(const SampleJob& j, long long piece) {
    const long long total = (long long)sample_rows(j) * j.ppr;
    if (piece < 0 || piece >= total) return;
    const int row = (int)(piece / j.ppr), part = (int)(piece % j.ppr);
    const RowRef rr = row_ref(j, row);
    const long long c0 = (long long)part * j.piece_len;
    const long long c1 = c0 + j.piece_len < j.V ? c0 + j.piece_len : j.V;
    const long long esz = j.f32 ? 4 : 2;
    const uintptr_t lo = (reinterpret_cast<uintptr_t>(rr.base) + (uintptr_t)(c0 * esz)) & ~(uintptr_t)15;
    const uintptr_t hi = (reinterpret_cast<uintptr_t>(rr.base) + (uintptr_t)(c1 * esz) + 15) & ~(uintptr_t)15;
    prefetch_l2_bulk(reinterpret_cast<const void*>(lo), (unsigned int)(hi - lo));
}

// Piece `piece` of the launch (piece / ppr is the row, piece % ppr its part);
// `next` is the piece this CTA takes after it (its bytes are prefetched to
// L2 now; -1: none).
static __device__ __noinline__ void sample_piece(const SampleJob& j, int piece, long long next, unsigned char* smem) {
    __shared__ unsigned int s_zmax, s_cnt;
    __shared__ int s_last, s_maxok;
    const int row = piece / j.ppr, part = piece % j.ppr;
    const RowRef rr = row_ref(j, row);
    const long long c0 = (long long)part * j.piece_len;
    const long long c1 = c0 + j.piece_len < j.V ? c0 + j.piece_len : j.V;
    int32_t* pen = reinterpret_cast<int32_t*>(smem);
    int2* buf = reinterpret_cast<int2*>(smem + kSampBitmapBytes);
    if (threadIdx.x == 0) {
        s_zmax = 0u;
        s_cnt = 0u;
        s_maxok = 0;
        prefetch_piece(j, next);
    }
    const int npen = load_penalty_list(j, rr.b, rr.i, pen);   // synchronises
    if (j.f32) piece_stream<float>(j, reinterpret_cast<const float*>(rr.base), c0, c1, &s_zmax, &s_cnt, buf);
    else piece_stream<uint16_t>(j, reinterpret_cast<const uint16_t*>(rr.base), c0, c1, &s_zmax, &s_cnt, buf);
    __syncthreads();
    // sort out the penalty set: its tokens leave the survivors (the finishing
    // CTA evaluates them exactly); the piece's maximum stands if an
    // unpenalised token reaches it
    const float Mz = key_max(s_zmax);
    const unsigned int n = s_cnt < (unsigned)kPieceBuf ? s_cnt : (unsigned)kPieceBuf;
    for (unsigned int t = threadIdx.x; t < n; t += blockDim.x) {
        int2 e = buf[t];
        if (npen > 0 && in_list(pen, npen, e.x)) {
            e.x = -1;
            buf[t] = e;
        } else if (__int_as_float(e.y) == Mz) {
            s_maxok = 1;
        }
    }
    __syncthreads();
    const bool redo = npen < 0 || s_cnt > (unsigned)kPieceBuf || (Mz > -INFINITY && !s_maxok);
    const float M = Mz > -INFINITY ? __fdiv_rn(Mz, j.temp) : -INFINITY;   // division is monotone
    const float thr = survive_thr(M, log_min_p(j));
    int2* rbuf = j.row_buf + (long long)row * j.rcap;
    if (!redo) {
        for (unsigned int t = threadIdx.x; t < n; t += blockDim.x) {
            const int2 e = buf[t];
            if (e.x < 0) continue;
            const float l = __fdiv_rn(__int_as_float(e.y), j.temp);
            if (l >= thr) {
                const unsigned int s = atomicAdd(j.row_cnt + row, 1u);
                if (s < (unsigned)j.rcap) rbuf[s] = make_int2(e.x, __float_as_int(l));
            }
        }
    }
    if (threadIdx.x == 0) {
        if (redo) atomicOr(j.row_ovf + row, 1u);
        else if (M > -INFINITY) atomicMax(j.row_max + row, ordered_key(M));
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        s_last = atomicAdd(j.row_done + row, 1u) == (unsigned)j.ppr - 1u;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    sample_finish_row(j, row, smem);
}

// ---------------------------------------------------------------------------
// a row's finishing CTA: exact min-p set, sort, top-p, then draw or hand over
// ---------------------------------------------------------------------------

// sort key: weight descending, then id ascending
__device__ __forceinline__ unsigned long long wid_key(float w, int id) {
    return ((unsigned long long)(~ordered_key(w)) << 32) | (uint32_t)id;
}

// Bitonic sort of keys[0, P) ascending, P a power of two.  Whole CTA.
__device__ __forceinline__ void bitonic_sort(unsigned long long* keys, unsigned int P) {
    for (unsigned int k = 2; k <= P; k <<= 1) {
        for (unsigned int jj = k >> 1; jj > 0; jj >>= 1) {
            for (unsigned int t = threadIdx.x; t < P; t += blockDim.x) {
                const unsigned int p2 = t ^ jj;
                if (p2 > t) {
                    const bool up = (t & k) == 0;
                    const unsigned long long x = keys[t], y = keys[p2];
                    if ((x > y) == up) {
                        keys[t] = y;
                        keys[p2] = x;
                    }
                }
            }
            __syncthreads();
        }
    }
}

// Sorts keys[0, n) ascending (keys distinct): by rank (each key counts the
// keys below it; one pass, tmp[n] holds the result until it is copied back)
// for n <= kRankSortMax, else bitonic over the next power of two (keys past
// n set to ~0 by the caller's padding here).  Whole CTA; synchronises.
__device__ __forceinline__ void sort_keys(unsigned long long* keys, unsigned int n, unsigned long long* tmp) {
    if (n <= (unsigned)kRankSortMax) {
        for (unsigned int t = threadIdx.x; t < n; t += blockDim.x) {
            const unsigned long long k = keys[t];
            unsigned int r = 0;
            for (unsigned int u = 0; u < n; ++u) r += keys[u] < k ? 1u : 0u;
            tmp[r] = k;
        }
        __syncthreads();
        for (unsigned int t = threadIdx.x; t < n; t += blockDim.x) keys[t] = tmp[t];
        __syncthreads();
        return;
    }
    unsigned int P = 1;
    while (P < n) P <<= 1;
    for (unsigned int t = n + threadIdx.x; t < P; t += blockDim.x) keys[t] = ~0ull;
    __syncthreads();
    bitonic_sort(keys, P);
}

// inverse-CDF pick: the first j with u * total < w_0 + ... + w_j, sums in
// order; n - 1 if none, 0 for an empty set
template <class WF>
__device__ __forceinline__ int pick_index_seq(int n, float total, float u, WF wfn) {
    const float target = __fmul_rn(u, total);
    float acc = 0.f;
    for (int t = 0; t < n; ++t) {
        acc = __fadd_rn(acc, wfn(t));
        if (target < acc) return t;
    }
    return n > 0 ? n - 1 : 0;
}

// Exact rescan of a whole row, used when a survivor buffer overflowed or a
// piece's maximum was held only by penalised tokens: pass 1 finds the row's
// largest scaled logit M, pass 2 keys every token with exp(l - M) >= min_p
// into keys (count in *cnt).  Whole CTA.
static __device__ __noinline__ float sample_rescan(const SampleJob& j, const RowRef& rr, uint32_t* bits,
                                                   unsigned long long* keys, unsigned int* cnt) {
    __shared__ unsigned int s_m;
    if (threadIdx.x == 0) s_m = 0u;
    float M = -INFINITY;
    for (int pass = 0; pass < 2; ++pass) {
        const float thr = pass == 0 ? INFINITY : survive_thr(M, log_min_p(j));
        for (long long c0 = 0; c0 < j.V; c0 += kPieceMax) {
            const long long c1 = c0 + kPieceMax < j.V ? c0 + kPieceMax : j.V;
            build_bitmap(j, rr.b, rr.i, c0, (int)((c1 - c0 + 31) / 32), bits);
            float mt = -INFINITY;
            for (long long x = c0 + threadIdx.x; x < c1; x += blockDim.x) {
                const long long rel = x - c0;
                const float z = row_elem(j, rr.base, x);
                const float l = ((bits[rel >> 5] >> (rel & 31)) & 1u) ? penalised_logit(j, z) : __fdiv_rn(z, j.temp);
                if (pass == 0) {
                    mt = fmaxf(mt, l);
                } else if (l >= thr) {
                    const float w = cand_weight(l, M);
                    if (w >= j.min_p) {
                        const unsigned int s = atomicAdd(cnt, 1u);
                        if (s < (unsigned)kCandCap) keys[s] = wid_key(w, (int)x);
                    }
                }
            }
            if (pass == 0) {
                mt = warp_max(mt);
                if ((threadIdx.x & 31) == 0 && mt > -INFINITY) atomicMax(&s_m, ordered_key(mt));
            }
            __syncthreads();
        }
        if (pass == 0) M = key_max(s_m);
        if (!(M > -INFINITY)) break;
    }
    return M;
}

// the sequence's walk (mode 0; defined below)
static __device__ void sample_walk(const SampleJob& j, int b, unsigned char* smem);

static __device__ void sample_finish_row(const SampleJob& j, int row, unsigned char* smem) {
    __shared__ unsigned int s_n, s_lp;
    __shared__ int s_keep, s_last;
    __shared__ float s_kept;
    uint32_t* bits = reinterpret_cast<uint32_t*>(smem);
    int32_t* pen = reinterpret_cast<int32_t*>(smem);
    unsigned long long* keys = reinterpret_cast<unsigned long long*>(smem + kSampBitmapBytes);
    float* wsh = reinterpret_cast<float*>(smem + kSampBitmapBytes + kSampKeyBytes);
    const RowRef rr = row_ref(j, row);
    const float Mnp = key_max(__ldcg(j.row_max + row));   // largest unpenalised scaled logit
    const unsigned int rc = __ldcg(j.row_cnt + row);
    bool ovf = __ldcg(j.row_ovf + row) != 0u || rc > (unsigned)j.rcap;
    if (threadIdx.x == 0) {
        s_n = 0u;
        s_lp = 0u;
    }
    __syncthreads();
    int npen = 0;
    if (!ovf) {
        npen = load_penalty_list(j, rr.b, rr.i, pen);   // synchronises
        ovf = npen < 0;
    }
    if (!ovf) {
        // the penalty set, each distinct token once, evaluated exactly
        float* plv = wsh;   // [npen] scaled logits (NaN: not a token of the set)
        for (int t = threadIdx.x; t < npen; t += blockDim.x) {
            const int x = pen[t];
            bool first = x >= 0 && x < j.V;
            for (int u = 0; u < t && first; ++u) first = pen[u] != x;
            float l = __int_as_float(0x7fc00000);
            if (first) l = penalised_logit(j, row_elem(j, rr.base, x));
            plv[t] = l;
            if (l == l) atomicMax(&s_lp, ordered_key(l));
        }
        __syncthreads();
        const float M = fmaxf(Mnp, key_max(s_lp));
        const float pre = survive_thr(M, log_min_p(j));   // cheap fp32 test before the exact weight
        if (M > -INFINITY) {
            const int2* rbuf = j.row_buf + (long long)row * j.rcap;
            for (unsigned int t = threadIdx.x; t < rc + (unsigned)npen; t += blockDim.x) {
                int x;
                float l;
                if (t < rc) {
                    const int2 e = __ldcg(rbuf + t);
                    x = e.x;
                    l = __int_as_float(e.y);
                } else {
                    x = pen[t - rc];
                    l = plv[t - rc];
                    if (!(l == l)) continue;
                }
                if (!(l >= pre)) continue;
                const float w = cand_weight(l, M);
                if (w >= j.min_p) {
                    const unsigned int s2 = atomicAdd(&s_n, 1u);
                    if (s2 < (unsigned)kCandCap) keys[s2] = wid_key(w, x);
                }
            }
        }
        __syncthreads();
    } else {
        sample_rescan(j, rr, bits, keys, &s_n);
    }
    unsigned int n = s_n;
    if (n > (unsigned)kCandCap) {
        if (threadIdx.x == 0) atomicCAS(&j.hdr->status, 0, MTP_ERR_CAPACITY);
        n = kCandCap;
    }
    __syncthreads();
    sort_keys(keys, n, reinterpret_cast<unsigned long long*>(smem));
    for (unsigned int t = threadIdx.x; t < n; t += blockDim.x) wsh[t] = key_to_float(~(uint32_t)(keys[t] >> 32));
    __syncthreads();
    if (threadIdx.x == 0) {
        int keep = (int)n;
        if (j.top_p < 1.f) {
            float tot = 0.f;
            for (unsigned int t = 0; t < n; ++t) tot = __fadd_rn(tot, wsh[t]);
            float cum = 0.f;
            for (unsigned int t = 0; t < n; ++t) {
                cum = __fadd_rn(cum, wsh[t]);
                if (__fdiv_rn(cum, tot) >= j.top_p) {
                    keep = (int)t + 1;
                    break;
                }
            }
        }
        float kept = 0.f;
        for (int t = 0; t < keep; ++t) kept = __fadd_rn(kept, wsh[t]);
        s_keep = keep;
        s_kept = kept;
        // the row's state is free again (every piece has finished)
        j.row_max[row] = 0u;
        j.row_cnt[row] = 0u;
        j.row_ovf[row] = 0u;
        j.row_done[row] = 0u;
    }
    __syncthreads();
    const int keep = s_keep;
    if (j.mode == 1) {
        if (threadIdx.x == 0) {
            const float u = philox_uniform(j.seed, j.offset, (uint32_t)rr.b, (uint32_t)rr.i, 0u);
            const int t = pick_index_seq(keep, s_kept, u, [&](int q) { return wsh[q]; });
            const int32_t tok = keep > 0 ? (int32_t)(uint32_t)(keys[t] & 0xFFFFFFFFull) : 0;
            if (j.out_draw) j.out_draw[(long long)rr.b * j.out_draw_ld + rr.i] = tok;
            if (j.out_amax) j.out_amax[rr.b] = (1ull << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)tok);
        }
        __syncthreads();
        return;
    }
    // mode 0: store the kept set, then count the row into its sequence
    for (int t = threadIdx.x; t < keep; t += blockDim.x) {
        j.keep_id[(long long)row * j.ccap + t] = (int32_t)(uint32_t)(keys[t] & 0xFFFFFFFFull);
        j.keep_w[(long long)row * j.ccap + t] = wsh[t];
    }
    if (threadIdx.x == 0) {
        j.n_keep[row] = keep;
        j.w_keep[row] = s_kept;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        s_last = atomicAdd(j.seq_done + rr.b, 1u) == (unsigned)(2 * j.N + 1) - 1u;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (threadIdx.x == 0) j.seq_done[rr.b] = 0u;
    sample_walk(j, rr.b, smem);
}

// ---------------------------------------------------------------------------
// the sequence's accept / residual / bonus walk (mode 0), one CTA
// ---------------------------------------------------------------------------

// Weight of token x in kept row `row` (0 if absent).  Whole CTA.
__device__ __forceinline__ float kept_weight(const SampleJob& j, int row, int32_t x, float* slot) {
    const int n = __ldcg(j.n_keep + row);
    if (threadIdx.x == 0) *slot = 0.f;
    __syncthreads();
    for (int t = threadIdx.x; t < n; t += blockDim.x)
        if (__ldcg(j.keep_id + (long long)row * j.ccap + t) == x) *slot = __ldcg(j.keep_w + (long long)row * j.ccap + t);
    __syncthreads();
    const float w = *slot;
    __syncthreads();
    return w;
}

static __device__ void sample_walk(const SampleJob& j, int b, unsigned char* smem) {
    __shared__ float s_slot;
    // q's kept set keyed by id (binary search), the residual weights
    unsigned long long* qk = reinterpret_cast<unsigned long long*>(smem + kSampBitmapBytes);
    float* rw = reinterpret_cast<float*>(smem + kSampBitmapBytes + kSampKeyBytes);
    const int R = j.N + 1;
    int32_t* out = j.out_tokens + (long long)b * R;
    int i = 0;
    for (; i < j.N; ++i) {
        const int trow = b * R + i, drow = j.B * R + b * j.N + i;
        const int32_t x = j.drafts[(long long)b * j.drafts_ld + i];
        const float Wt = __ldcg(j.w_keep + trow), Wd = __ldcg(j.w_keep + drow);
        const float wpx = kept_weight(j, trow, x, &s_slot), wqx = kept_weight(j, drow, x, &s_slot);
        // p(x) and q(x) divide only when x is kept (0 otherwise)
        const float px = wpx > 0.f || wpx < 0.f ? __fdiv_rn(wpx, Wt) : 0.f;
        const float qx = wqx > 0.f || wqx < 0.f ? __fdiv_rn(wqx, Wd) : 0.f;
        const float u = philox_uniform(j.seed, j.offset, (uint32_t)b, (uint32_t)i, 1u);
        if (u < __fdiv_rn(px, qx)) {
            if (threadIdx.x == 0) out[i] = x;
            continue;
        }
        // residual max(p - q, 0) over p's kept set in p's order
        const int np = __ldcg(j.n_keep + trow), nq = __ldcg(j.n_keep + drow);
        for (int t = threadIdx.x; t < nq; t += blockDim.x) {
            const int32_t id = __ldcg(j.keep_id + (long long)drow * j.ccap + t);
            const float w = __ldcg(j.keep_w + (long long)drow * j.ccap + t);
            qk[t] = ((unsigned long long)(uint32_t)id << 32) | __float_as_uint(w);
        }
        __syncthreads();
        sort_keys(qk, (unsigned)nq, reinterpret_cast<unsigned long long*>(smem));
        for (int t = threadIdx.x; t < np; t += blockDim.x) {
            const uint32_t id = (uint32_t)__ldcg(j.keep_id + (long long)trow * j.ccap + t);
            const float pj = __fdiv_rn(__ldcg(j.keep_w + (long long)trow * j.ccap + t), Wt);
            int lo = 0, hi = nq;   // first index with id >= this id
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if ((uint32_t)(qk[mid] >> 32) < id) lo = mid + 1;
                else hi = mid;
            }
            float qj = 0.f;
            if (lo < nq && (uint32_t)(qk[lo] >> 32) == id) qj = __fdiv_rn(__uint_as_float((uint32_t)qk[lo]), Wd);
            rw[t] = pj > qj ? __fsub_rn(pj, qj) : 0.f;
        }
        __syncthreads();
        float Rt = 0.f;
        if (threadIdx.x == 0)
            for (int t = 0; t < np; ++t) Rt = __fadd_rn(Rt, rw[t]);
        if (threadIdx.x == 0) s_slot = Rt;
        __syncthreads();
        Rt = s_slot;
        if (!(Rt > 0.f)) {   // p == q on p's support: the residual is empty, draw from p
            for (int t = threadIdx.x; t < np; t += blockDim.x) rw[t] = __ldcg(j.keep_w + (long long)trow * j.ccap + t);
            __syncthreads();
        }
        if (threadIdx.x == 0) {
            const float u2 = philox_uniform(j.seed, j.offset, (uint32_t)b, (uint32_t)i, 2u);
            const int t = pick_index_seq(np, Rt > 0.f ? Rt : Wt, u2, [&](int q) { return rw[q]; });
            out[i] = np > 0 ? __ldcg(j.keep_id + (long long)trow * j.ccap + t) : 0;
        }
        __syncthreads();
        break;
    }
    if (i == j.N) {   // every draft accepted: the bonus token from p_N
        const int trow = b * R + j.N;
        const long long tb = (long long)trow * j.ccap;
        const int np = __ldcg(j.n_keep + trow);
        for (int t = threadIdx.x; t < np; t += blockDim.x) rw[t] = __ldcg(j.keep_w + tb + t);
        __syncthreads();
        if (threadIdx.x == 0) {
            const float u3 = philox_uniform(j.seed, j.offset, (uint32_t)b, (uint32_t)j.N, 3u);
            const int t = pick_index_seq(np, __ldcg(j.w_keep + trow), u3, [&](int q) { return rw[q]; });
            out[j.N] = np > 0 ? __ldcg(j.keep_id + tb + t) : 0;
        }
    }
    if (threadIdx.x == 0) {
        for (int t = i + 1; t < R; ++t) out[t] = -1;
        j.out_n_accept[b] = i;
    }
    __syncthreads();
}

}  // namespace mtp
