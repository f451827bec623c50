// draft_bf16_tc.cu -- bf16 instantiations of the persistent draft-block
// kernel with the tensor-core LM head and projections (batched launches).
#include "draft_kernel.cuh"

namespace mtp {

cudaError_t launch_draft_bf16_tc(const DraftParams& p, int grid, size_t smem, cudaStream_t s) {
    switch (p.hd) {
    case 64: return launch_draft_t<uint16_t, 64, true>(p, grid, smem, s);
    case 128: return launch_draft_t<uint16_t, 128, true>(p, grid, smem, s);
    case 256: return launch_draft_t<uint16_t, 256, true>(p, grid, smem, s);
    case 512: return launch_draft_t<uint16_t, 512, true>(p, grid, smem, s);
    default: return launch_draft_t<uint16_t, 32, true>(p, grid, smem, s);
    }
}

int draft_blocks_per_sm_bf16_tc(int hd, size_t smem) {
    switch (hd) {
    case 64: return draft_blocks_per_sm_t<uint16_t, 64, true>(smem);
    case 128: return draft_blocks_per_sm_t<uint16_t, 128, true>(smem);
    case 256: return draft_blocks_per_sm_t<uint16_t, 256, true>(smem);
    case 512: return draft_blocks_per_sm_t<uint16_t, 512, true>(smem);
    default: return draft_blocks_per_sm_t<uint16_t, 32, true>(smem);
    }
}

}  // namespace mtp
