// draft_inst.cu -- one instantiation of the persistent draft-block kernel.
//
// The build compiles this file once per (weight type, head dimension,
// tensor-core paths) combination, selected by MTP_WT_BF16, MTP_HD and
// MTP_TC (and MTP_Q8 / MTP_Q4: Q8_0 / Q4_0 projections beside a bf16 table and KV), so the
// kernel variants compile in parallel processes.  Each
// object defines launch_draft_<variant> and draft_blocks_per_sm_<variant>;
// draft_dispatch.cu picks one at run time.
#include "draft_kernel.cuh"

#if !defined(MTP_WT_BF16) || !defined(MTP_HD) || !defined(MTP_TC)
#error "draft_inst.cu needs MTP_WT_BF16, MTP_HD and MTP_TC"
#endif

#define MTP_CAT2(a, b) a##b
#define MTP_CAT(a, b) MTP_CAT2(a, b)
#if !defined(MTP_Q8)
#define MTP_Q8 0
#endif
#if !defined(MTP_Q4)
#define MTP_Q4 0
#endif
#if MTP_Q8
#define MTP_WT uint16_t
#define MTP_PT int8_t
#define MTP_VAR MTP_CAT(q8_, MTP_HD)
#elif MTP_Q4
#define MTP_WT uint16_t
#define MTP_PT Q4Code
#define MTP_VAR MTP_CAT(q4_, MTP_HD)
#elif MTP_WT_BF16
#define MTP_WT uint16_t
#if MTP_TC
#define MTP_VAR MTP_CAT(bf16_tc_, MTP_HD)
#else
#define MTP_VAR MTP_CAT(bf16_cc_, MTP_HD)
#endif
#else
#define MTP_WT float
#define MTP_VAR MTP_CAT(f32_, MTP_HD)
#endif
#ifndef MTP_PT
#define MTP_PT MTP_WT
#endif

namespace mtp {

cudaError_t MTP_CAT(launch_draft_, MTP_VAR)(const DraftParams& p, int grid, size_t smem, cudaStream_t s) {
    return launch_draft_t<MTP_WT, MTP_HD, (MTP_TC != 0), MTP_PT>(p, grid, smem, s);
}

int MTP_CAT(draft_blocks_per_sm_, MTP_VAR)(size_t smem) {
    return draft_blocks_per_sm_t<MTP_WT, MTP_HD, (MTP_TC != 0), MTP_PT>(smem);
}

}  // namespace mtp
