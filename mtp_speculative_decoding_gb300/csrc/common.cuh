// common.cuh -- device helpers shared by the draft and verify kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "mtp.h"

namespace mtp {

constexpr int kThreads = 512;          // threads per CTA of every kernel here
constexpr int kWarps = kThreads / 32;

// ---------------------------------------------------------------------------
// workspace header (first 256 bytes of every workspace; zeroed per call)
// ---------------------------------------------------------------------------
struct WsHeader {
    unsigned int barrier;     // grid-barrier arrival counter
    int status;               // MTP_OK or a device-side MTP_ERR_* code
    unsigned int done;        // last-arriver counters of single-launch kernels
    unsigned int pad[61];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

// ---------------------------------------------------------------------------
// loads
// ---------------------------------------------------------------------------

// 16-byte streaming load of read-only data (weights, logits, KV): no L1
// allocation, 256-byte L2 prefetch hint.
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}
// L2 policy: evict first (weight streams)
__device__ __forceinline__ unsigned long long l2_evict_first() {
    unsigned long long pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
// ld_stream16 for weight streams read once per step, under an L2 policy
// from l2_evict_first(): the lines go first when L2 evicts, so the small
// vectors, gains and split partials that phases re-read keep
// their places
__device__ __forceinline__ uint4 ld_weight16(const void* p, unsigned long long pol) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.L2::cache_hint.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p), "l"(pol));
    return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }

// element i of a weight/KV/logit array of either dtype, as fp32
template <typename WT> __device__ __forceinline__ float ld_elem(const WT* p, long long i);
template <> __device__ __forceinline__ float ld_elem<float>(const float* p, long long i) { return __ldg(p + i); }
template <> __device__ __forceinline__ float ld_elem<uint16_t>(const uint16_t* p, long long i) {
    return bf16_to_f32(__ldg(p + i));
}

// 16-byte asynchronous global -> shared copies (L2 only), grouped by commit
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                     static_cast<unsigned int>(__cvta_generic_to_shared(smem_dst))),
                 "l"(gsrc)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// mbarrier + bulk (TMA) copy primitives
__device__ __forceinline__ unsigned int smem_addr(const void* p) {
    return static_cast<unsigned int>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(unsigned long long* bar, unsigned int count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ void mbar_arrive_expect_tx(unsigned long long* bar, unsigned int bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(unsigned long long* bar, unsigned int parity) {
    unsigned int ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// global -> shared bulk copy completing on `bar`; addresses 16-byte aligned, bytes a multiple of 16
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, unsigned int bytes, unsigned long long* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}
// bulk_g2s with an L2 cache policy
__device__ __forceinline__ void bulk_g2s_pol(void* dst, const void* src, unsigned int bytes, unsigned long long* bar,
                                             unsigned long long pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(pol)
        : "memory");
}
// bulk prefetch of [p, p + bytes) into L2 (p 16-byte aligned, bytes a multiple of 16)
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, unsigned int bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
// bulk copy shared -> global (both 16-byte aligned, bytes a multiple of 16),
// tracked by the issuing thread's bulk groups
__device__ __forceinline__ void bulk_s2g(void* gdst, const void* ssrc, unsigned int bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(smem_addr(ssrc)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// this thread's bulk stores have read their shared-memory sources
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// this thread's bulk stores are complete (their global writes performed)
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// L2 prefetch of one box of a 2-D tensor map
__device__ __forceinline__ void tma_prefetch_2d(const void* tmap, int x, int y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(tmap), "r"(x), "r"(y)
                 : "memory");
}
// order earlier generic-proxy shared-memory accesses before later bulk-copy writes
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// plain arrive (count 1) on an mbarrier
__device__ __forceinline__ void mbar_arrive(unsigned long long* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
// order this thread's earlier generic-proxy global writes before later
// async-proxy (tensor copy) reads of them
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

// 2-D tiled tensor copy global -> shared through a tensor map (generic
// address of a __grid_constant__ parameter) under an L2 cache policy; x is
// the innermost coordinate
__device__ __forceinline__ void tma_load_2d_pol(void* dst, const void* tmap, int x, int y, unsigned long long* bar,
                                                unsigned long long pol) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
        "%3}], [%4], %5;" ::"r"(smem_addr(dst)),
        "l"(tmap), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(pol)
        : "memory");
}

// ---------------------------------------------------------------------------
// 5th-generation tensor cores: tensor memory, MMA, commit, loads
// ---------------------------------------------------------------------------
// whole warp: allocate ncols (power of 2, >= 32) tensor-memory columns; the
// base address is written to *dst
__device__ __forceinline__ void tmem_alloc(unsigned int* dst, unsigned int ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst)), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(unsigned int taddr, unsigned int ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, bf16 inputs, fp32 accumulate
__device__ __forceinline__ void umma_bf16(unsigned int d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// arrive once on `bar` when every MMA this thread issued so far has completed
__device__ __forceinline__ void umma_commit(unsigned long long* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}
// 16 consecutive fp32 columns of this thread's tensor-memory lane
__device__ __forceinline__ void tmem_ld16(unsigned int taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, "
        "[%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor of a K-major operand tile whose rows are
// 128 bytes (64 bf16) written by a tensor copy with 128-byte swizzle; the
// tile starts on a 1024-byte boundary (8-row groups 1024 bytes apart).
// Advancing the start by 32 bytes selects the next 16-element K slice.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t smem_byte_addr) {
    uint64_t d = 0;
    d |= (uint64_t)((smem_byte_addr >> 4) & 0x3FFFu);   // start address
    d |= (uint64_t)1 << 16;                              // leading offset (unused with 128-byte swizzle)
    d |= (uint64_t)(1024 >> 4) << 32;                    // stride offset: 8 rows x 128 bytes
    d |= (uint64_t)1 << 46;                              // descriptor version
    d |= (uint64_t)2 << 61;                              // 128-byte swizzle
    return d;
}
// instruction descriptor: bf16 A and B (K-major), fp32 D, shape M x N
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ---------------------------------------------------------------------------
// reductions
// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
        v = w > v ? w : v;
    }
    return v;
}

// Sum over the CTA; every thread gets the result.  `red` is kWarps floats of
// shared scratch; the function synchronizes the CTA twice.
__device__ __forceinline__ float block_sum(float v, float* red) {
    v = warp_sum(v);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float t = lane < kWarps ? red[lane] : 0.f;
    return warp_sum(t);
}

// ---------------------------------------------------------------------------
// argmax keys: a total order on (value, index) packed into 64 bits so that an
// unsigned max picks the largest value and, among equal values, the lowest
// index.  NaN orders below -inf (never wins); -0 and +0 are equal.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t ordered_key(float f) {
    if (f != f) return 0u;
    uint32_t u = __float_as_uint(f);
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ unsigned long long pack_argmax(float v, uint32_t idx) {
    return ((unsigned long long)ordered_key(v) << 32) | (unsigned long long)(0xFFFFFFFFu - idx);
}
__device__ __forceinline__ uint32_t unpack_index(unsigned long long p) {
    return 0xFFFFFFFFu - (uint32_t)(p & 0xFFFFFFFFull);
}

// ---------------------------------------------------------------------------
// Philox-4x32-10 (Salmon et al., SC'11): 10 rounds of the 4x32 bijection with
// multipliers 0xD2511F53 / 0xCD9E8D57 and Weyl key increments 0x9E3779B9 /
// 0xBB67AE85.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint2 k) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
        const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
        c = make_uint4(hi1 ^ c.y ^ k.x, lo1, hi0 ^ c.w ^ k.y, lo0);
        k.x += 0x9E3779B9u;
        k.y += 0xBB67AE85u;
    }
    return c;
}

// uniform in [0, 1) for (sequence b, row i, purpose): 24 random bits, exact in fp32
__device__ __forceinline__ float philox_uniform(unsigned long long seed, unsigned long long offset,
                                                uint32_t b, uint32_t i, uint32_t purpose) {
    uint4 c = make_uint4(b, i * 4u + purpose, (uint32_t)offset, (uint32_t)(offset >> 32));
    uint2 k = make_uint2((uint32_t)seed, (uint32_t)(seed >> 32));
    uint4 o = philox4x32_10(c, k);
    return (float)(o.x >> 8) * (1.0f / 16777216.0f);
}

// ---------------------------------------------------------------------------
// grid barrier with a time limit
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ unsigned int ld_acquire(const unsigned int* p) {
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ int ld_relaxed(const int* p) {
    int v;
    asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Every CTA of a co-resident (cooperative) grid calls this the same number of
// times.  `epoch` counts barriers passed by the calling CTA (thread 0's copy is
// the one used).  The counter starts at 0 (the host zeroes the header before
// the launch).  A CTA that waits longer than `limit_ns`, or sees a non-zero
// status, gives up: it records MTP_ERR_TIMEOUT (first writer wins) and returns
// false, after which the caller must return without touching shared results.
__device__ __forceinline__ bool grid_barrier(WsHeader* hdr, unsigned int& epoch, unsigned long long limit_ns,
                                             unsigned int arrivals_per_epoch) {
    __shared__ int s_ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        epoch += 1;
        const unsigned int target = epoch * arrivals_per_epoch;
        // release: the CTA's writes (ordered before by the CTA barrier) are
        // visible at GPU scope before its arrival; the acquire load that sees
        // every arrival orders the CTA's later reads after them
        asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(&hdr->barrier), "r"(1u) : "memory");
        const unsigned long long t0 = global_ns();
        int ok = 1;
        unsigned int spins = 0;
        while (true) {
            const unsigned int v = ld_acquire(&hdr->barrier);
            if ((int)(v - target) >= 0) break;
            if ((++spins & 63u) == 0) {   // error status and time limit, every 64 polls
                if (ld_relaxed(&hdr->status) != 0) { ok = 0; break; }
                if (global_ns() - t0 > limit_ns) {
                    atomicCAS(&hdr->status, 0, MTP_ERR_TIMEOUT);
                    ok = 0;
                    break;
                }
            }
        }
        s_ok = ok;
    }
    __syncthreads();
    return s_ok != 0;
}

}  // namespace mtp
