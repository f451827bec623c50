// draft_bf16.cu -- bf16 instantiations of the persistent draft-block kernel
// without the tensor-core paths (batches below the tensor-core threshold).
#include "draft_kernel.cuh"

namespace mtp {

cudaError_t launch_draft_bf16_cc(const DraftParams& p, int grid, size_t smem, cudaStream_t s) {
    switch (p.hd) {
    case 64: return launch_draft_t<uint16_t, 64, false>(p, grid, smem, s);
    case 128: return launch_draft_t<uint16_t, 128, false>(p, grid, smem, s);
    case 256: return launch_draft_t<uint16_t, 256, false>(p, grid, smem, s);
    case 512: return launch_draft_t<uint16_t, 512, false>(p, grid, smem, s);
    default: return launch_draft_t<uint16_t, 32, false>(p, grid, smem, s);
    }
}

int draft_blocks_per_sm_bf16_cc(int hd, size_t smem) {
    switch (hd) {
    case 64: return draft_blocks_per_sm_t<uint16_t, 64, false>(smem);
    case 128: return draft_blocks_per_sm_t<uint16_t, 128, false>(smem);
    case 256: return draft_blocks_per_sm_t<uint16_t, 256, false>(smem);
    case 512: return draft_blocks_per_sm_t<uint16_t, 512, false>(smem);
    default: return draft_blocks_per_sm_t<uint16_t, 32, false>(smem);
    }
}

}  // namespace mtp
