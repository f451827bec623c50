// noalloc.cu -- greedy verify for callers that cannot hand the library a
// workspace.
//
// mtp_verify_greedy needs a little scratch (a 256-byte header and one 8-byte
// argmax slot per verified row).  This variant keeps that scratch in a
// file-scope device array instead of a caller buffer, so it works for callers
// that are not allowed to allocate device memory.  The array is small and
// fixed: every GPU that loads the library holds it until the process exits.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "common.cuh"
#include "mtp.h"
#include "verify.cuh"

namespace {

constexpr size_t kScratchBytes = 4096;   // header (256 B) + 480 argmax slots

// The scratch itself.  In host code this name is only a stand-in for the
// device symbol: its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_verify_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {nullptr};
int g_sms[kMaxDevices] = {0};

// Device address of the scratch and the SM count of the current device; the
// first call on a device looks them up (with that device current).
int device_scratch(void** addr, int* sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MTP_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_verify_scratch) != cudaSuccess || p == nullptr) return MTP_ERR_CUDA;
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            return MTP_ERR_CUDA;
        g_sms[dev] = n;
        g_scratch_addr[dev] = p;
    }
    *addr = g_scratch_addr[dev];
    *sms = g_sms[dev];
    return MTP_OK;
}

}  // namespace

extern "C" int mtp_verify_greedy_noalloc(const void* logits, int ldtype, int B, int N, int V,
                                         const int32_t* drafts, int32_t* out_tokens, int32_t* out_n_accept,
                                         mtp_stream_t stream) {
    if (!logits || !out_tokens || !out_n_accept) return MTP_ERR_ARG;
    if (B < 1 || B > MTP_MAX_BATCH || N < 0 || N > 16 || V < 1) return MTP_ERR_ARG;
    if (N > 0 && !drafts) return MTP_ERR_ARG;
    if (ldtype != MTP_DTYPE_F32 && ldtype != MTP_DTYPE_BF16) return MTP_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(logits) & (ldtype == MTP_DTYPE_BF16 ? 1 : 3)) != 0) return MTP_ERR_ARG;
    const size_t need = sizeof(mtp::WsHeader) + (size_t)B * (N + 1) * sizeof(unsigned long long);
    if (need > kScratchBytes) return MTP_ERR_UNSUPPORTED;   // B * (1 + N) above 480 rows
    void* base = nullptr;
    int sms = 0;
    const int rc = device_scratch(&base, &sms);
    if (rc != MTP_OK) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // the header's counter and the argmax slots must start at zero on every call
    if (cudaMemsetAsync(base, 0, need, s) != cudaSuccess) return MTP_ERR_CUDA;
    mtp::VerifyGreedyArgs a;
    a.logits = logits;
    a.B = B;
    a.N = N;
    a.V = V;
    a.drafts = drafts;
    a.out_tokens = out_tokens;
    a.out_n_accept = out_n_accept;
    a.hdr = static_cast<mtp::WsHeader*>(base);
    a.amax = reinterpret_cast<unsigned long long*>(static_cast<char*>(base) + sizeof(mtp::WsHeader));
    return mtp::launch_verify_greedy(a, ldtype, sms, s) == cudaSuccess ? MTP_OK : MTP_ERR_CUDA;
}
