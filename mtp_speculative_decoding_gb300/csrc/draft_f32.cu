// draft_f32.cu -- fp32 instantiations of the persistent draft-block kernel.
#include "draft_kernel.cuh"

namespace mtp {

cudaError_t launch_draft_f32(const DraftParams& p, int grid, size_t smem, cudaStream_t s) {
    switch (p.hd) {
    case 64: return launch_draft_t<float, 64, false>(p, grid, smem, s);
    case 128: return launch_draft_t<float, 128, false>(p, grid, smem, s);
    case 256: return launch_draft_t<float, 256, false>(p, grid, smem, s);
    case 512: return launch_draft_t<float, 512, false>(p, grid, smem, s);
    default: return launch_draft_t<float, 32, false>(p, grid, smem, s);
    }
}

int draft_blocks_per_sm_f32(int hd, size_t smem) {
    switch (hd) {
    case 64: return draft_blocks_per_sm_t<float, 64, false>(smem);
    case 128: return draft_blocks_per_sm_t<float, 128, false>(smem);
    case 256: return draft_blocks_per_sm_t<float, 256, false>(smem);
    case 512: return draft_blocks_per_sm_t<float, 512, false>(smem);
    default: return draft_blocks_per_sm_t<float, 32, false>(smem);
    }
}

// A grid barrier whose arrival count can never be reached: every CTA waits
// until its time limit, records MTP_ERR_TIMEOUT and returns.
__global__ void __launch_bounds__(kThreads, 1) barrier_timeout_probe(WsHeader* hdr, unsigned long long limit_ns) {
    unsigned int epoch = 0;
    grid_barrier(hdr, epoch, limit_ns, gridDim.x + 1u);
}

cudaError_t launch_barrier_timeout_probe(WsHeader* hdr, unsigned long long limit_ns, cudaStream_t s) {
    void* args[] = {&hdr, &limit_ns};
    return cudaLaunchCooperativeKernel((const void*)barrier_timeout_probe, dim3(2), dim3(kThreads), args, 0, s);
}

}  // namespace mtp
