// draft_dispatch.cu -- run-time choice of the draft-kernel variant (weight
// type, head dimension, tensor-core paths) among the objects built from
// draft_inst.cu, and the grid-barrier time-out probe.
#include "draft.cuh"

namespace mtp {

#define MTP_DECL_VARIANT(v)                                                                   \
    cudaError_t launch_draft_##v(const DraftParams& p, int grid, size_t smem, cudaStream_t s); \
    int draft_blocks_per_sm_##v(size_t smem);
#define MTP_DECL_HDS(pfx) \
    MTP_DECL_VARIANT(pfx##32) MTP_DECL_VARIANT(pfx##64) MTP_DECL_VARIANT(pfx##128) MTP_DECL_VARIANT(pfx##256) MTP_DECL_VARIANT(pfx##512)
MTP_DECL_HDS(f32_)
MTP_DECL_HDS(bf16_cc_)
MTP_DECL_HDS(bf16_tc_)
MTP_DECL_VARIANT(q8_64) MTP_DECL_VARIANT(q8_128) MTP_DECL_VARIANT(q8_256)
MTP_DECL_VARIANT(q4_64) MTP_DECL_VARIANT(q4_128) MTP_DECL_VARIANT(q4_256)

#define MTP_SWITCH_HD(pfx, call)        \
    switch (hd) {                       \
    case 64: return pfx##64 call;       \
    case 128: return pfx##128 call;     \
    case 256: return pfx##256 call;     \
    case 512: return pfx##512 call;     \
    default: return pfx##32 call;       \
    }

cudaError_t launch_draft_f32(const DraftParams& p, int grid, size_t smem, cudaStream_t s) {
    const int hd = p.hd;
    MTP_SWITCH_HD(launch_draft_f32_, (p, grid, smem, s))
}
cudaError_t launch_draft_bf16_cc(const DraftParams& p, int grid, size_t smem, cudaStream_t s) {
    const int hd = p.hd;
    MTP_SWITCH_HD(launch_draft_bf16_cc_, (p, grid, smem, s))
}
cudaError_t launch_draft_bf16_tc(const DraftParams& p, int grid, size_t smem, cudaStream_t s) {
    const int hd = p.hd;
    MTP_SWITCH_HD(launch_draft_bf16_tc_, (p, grid, smem, s))
}
cudaError_t launch_draft_q8(const DraftParams& p, int grid, size_t smem, cudaStream_t s) {
    switch (p.hd) {
    case 64: return launch_draft_q8_64(p, grid, smem, s);
    case 128: return launch_draft_q8_128(p, grid, smem, s);
    default: return launch_draft_q8_256(p, grid, smem, s);
    }
}
int draft_blocks_per_sm_q8(int hd, size_t smem) {
    switch (hd) {
    case 64: return draft_blocks_per_sm_q8_64(smem);
    case 128: return draft_blocks_per_sm_q8_128(smem);
    default: return draft_blocks_per_sm_q8_256(smem);
    }
}
cudaError_t launch_draft_q4(const DraftParams& p, int grid, size_t smem, cudaStream_t s) {
    switch (p.hd) {
    case 64: return launch_draft_q4_64(p, grid, smem, s);
    case 128: return launch_draft_q4_128(p, grid, smem, s);
    default: return launch_draft_q4_256(p, grid, smem, s);
    }
}
int draft_blocks_per_sm_q4(int hd, size_t smem) {
    switch (hd) {
    case 64: return draft_blocks_per_sm_q4_64(smem);
    case 128: return draft_blocks_per_sm_q4_128(smem);
    default: return draft_blocks_per_sm_q4_256(smem);
    }
}
int draft_blocks_per_sm_f32(int hd, size_t smem) { MTP_SWITCH_HD(draft_blocks_per_sm_f32_, (smem)) }
int draft_blocks_per_sm_bf16_cc(int hd, size_t smem) { MTP_SWITCH_HD(draft_blocks_per_sm_bf16_cc_, (smem)) }
int draft_blocks_per_sm_bf16_tc(int hd, size_t smem) { MTP_SWITCH_HD(draft_blocks_per_sm_bf16_tc_, (smem)) }

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
