// verify.cu -- verify-accept kernels.
//
// Greedy ("MTP decoding (--mtp)", How it is wired): one launch.  The (1+N)
// rows of every sequence are split into V-chunks; each CTA reduces its chunk
// to a packed (value, index) key and folds it into the row's slot with one
// 64-bit atomicMax, so the result does not depend on CTA order.  The last CTA
// to finish (a counter in the workspace header) turns the row argmaxes into
// the accepted prefix and the bonus token.
//
// Exact sampling ("opus-mtp-turbo: Track 1 report", item 4): one plain
// launch over pieces of every target and draft row; one pass over the
// logits, the rows' finishing CTAs build the kept sets and the sequences'
// finishing CTAs take the accept / residual / bonus decisions (sample.cuh).
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
    const int split = a.split;
    const int row = (int)(blockIdx.x / (unsigned)split);   // b * (1+N) + i
    const long long V = a.V;
    const long long chunk = (V + split - 1) / split;
    const long long c0 = (long long)(blockIdx.x % (unsigned)split) * chunk;
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
        const unsigned int total = gridDim.x;
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
    VerifyGreedyArgs b = a;
    b.split = (int)split;
    const unsigned int grid = (unsigned int)(split * rows);
    if (ldtype == MTP_DTYPE_BF16)
        verify_greedy_kernel<uint16_t><<<grid, 256, 0, s>>>(b);
    else
        verify_greedy_kernel<float><<<grid, 256, 0, s>>>(b);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// sampling: exact speculative verification and draft draws (sample.cuh)
// ---------------------------------------------------------------------------

constexpr int kSampThreads = 256;

// Persistent over the pieces: CTA c starts with piece c, then takes the next
// unclaimed piece from a counter (CTAs that finish a row or a sequence on the
// way simply take fewer pieces), and prefetches that next piece into L2
// while it works on the current one.
__global__ void __launch_bounds__(kSampThreads, 3) sample_kernel(const __grid_constant__ SampleJob j) {
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ long long s_next;
    const long long total = (long long)sample_rows(j) * j.ppr;
    long long cur = blockIdx.x;
    if (threadIdx.x == 0) prefetch_piece(j, cur);
    while (cur < total) {
        if (threadIdx.x == 0) s_next = (long long)gridDim.x + atomicAdd(j.next_piece, 1u);
        __syncthreads();
        const long long nxt = s_next;   // read before sample_piece's first barrier; rewritten only after it
        sample_piece(j, (int)cur, nxt < total ? nxt : -1, smem);
        cur = nxt;
    }
}

void sample_piece_plan(long long V, long long rows, int grid, int* ppr, int* piece_len) {
    long long lo = (V + kPieceMax - 1) / kPieceMax;   // pieces fit the bitmap
    long long hi = V / 2048 > lo ? V / 2048 : lo;       // pieces of at least ~2K tokens
    long long want = (2LL * grid + rows - 1) / rows;    // about two pieces per CTA
    long long n = want < lo ? lo : (want > hi ? hi : want);
    long long len = (V + n - 1) / n;
    len = (len + 255) & ~255LL;
    if (len > kPieceMax) len = kPieceMax;
    if (len < 256) len = 256;
    *piece_len = (int)len;
    *ppr = (int)((V + len - 1) / len);
}

// The kernel's shared-memory attribute and occupancy, once per device.
namespace {
constexpr int kMaxDev = 64;
int g_samp_ready[kMaxDev] = {0};
int g_samp_per_sm[kMaxDev] = {0};
int sample_setup() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return -1;
    if (!g_samp_ready[dev]) {
        if (cudaFuncSetAttribute(sample_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSampleSmem) !=
            cudaSuccess)
            return -1;
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, sample_kernel, kSampThreads, kSampleSmem) != cudaSuccess)
            return -1;
        g_samp_per_sm[dev] = n;
        g_samp_ready[dev] = 1;
    }
    return dev;
}
}  // namespace

cudaError_t launch_sample(const SampleJob& j, int sms, cudaStream_t s) {
    const int dev = sample_setup();
    if (dev < 0) return cudaErrorInvalidValue;
    const long long total = (long long)sample_rows(j) * j.ppr;
    const long long resident = (long long)(g_samp_per_sm[dev] > 0 ? g_samp_per_sm[dev] : 1) * (sms > 0 ? sms : 1);
    const unsigned int grid = (unsigned int)(total < resident ? total : resident);
    sample_kernel<<<grid, kSampThreads, kSampleSmem, s>>>(j);
    return cudaGetLastError();
}

int sample_blocks_per_sm() {
    const int dev = sample_setup();
    return dev < 0 ? 0 : g_samp_per_sm[dev];
}

}  // namespace mtp
