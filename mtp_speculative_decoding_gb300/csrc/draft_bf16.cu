// draft_bf16.cu -- bf16 instantiations of the persistent draft-block kernel.
#include "draft_kernel.cuh"

namespace mtp {

cudaError_t launch_draft_bf16(const DraftParams& p, int grid, size_t smem, cudaStream_t s) {
    switch (p.hd) {
    case 64: return launch_draft_t<uint16_t, 64>(p, grid, smem, s);
    case 128: return launch_draft_t<uint16_t, 128>(p, grid, smem, s);
    case 256: return launch_draft_t<uint16_t, 256>(p, grid, smem, s);
    case 512: return launch_draft_t<uint16_t, 512>(p, grid, smem, s);
    default: return launch_draft_t<uint16_t, 32>(p, grid, smem, s);
    }
}

int draft_blocks_per_sm_bf16(int hd, size_t smem) {
    switch (hd) {
    case 64: return draft_blocks_per_sm_t<uint16_t, 64>(smem);
    case 128: return draft_blocks_per_sm_t<uint16_t, 128>(smem);
    case 256: return draft_blocks_per_sm_t<uint16_t, 256>(smem);
    case 512: return draft_blocks_per_sm_t<uint16_t, 512>(smem);
    default: return draft_blocks_per_sm_t<uint16_t, 32>(smem);
    }
}

}  // namespace mtp
