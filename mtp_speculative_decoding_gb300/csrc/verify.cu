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
#include "sample.cuh"
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
// exact sampling (device functions in sample.cuh)
// ---------------------------------------------------------------------------

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
