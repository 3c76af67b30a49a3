// gdn_tc.cuh -- fifth-generation tensor core (tcgen05) building blocks for
// sm_103a: tensor-memory allocation, shared-memory matrix descriptors, the
// instruction descriptor of a TF32 MMA with fp32 accumulation, MMA issue with
// the operand A in shared or tensor memory, commit to an mbarrier with a
// bounded wait, and warp-wide tensor-memory loads and stores.  Inline PTX
// written from the PTX ISA's description of these instructions.
//
// Operand layout used throughout: K-major with the 128-byte swizzle.  A tile
// of R rows x K fp32 elements is stored as K/32 column blocks of R rows x 128
// bytes; inside a block, row r's 16-byte chunk j sits at r*128 + ((j ^ (r%8))
// * 16).  Blocks start on 1024-byte boundaries, eight rows (one swizzle atom)
// are 1024 bytes apart, and one MMA (K = 8 fp32 = 32 bytes) starts 32 bytes
// further into the block for each step along K.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {
namespace tc {

// ---------------------------------------------------------------- descriptors

// Shared-memory matrix descriptor: start address, leading and stride byte
// offsets (16-byte units), descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t smem_addr)
{
    return (uint64_t)((smem_addr & 0x3FFFFu) >> 4)        // start address
         | ((uint64_t)1 << 16)                            // leading byte offset (unused with this swizzle)
         | ((uint64_t)(1024 >> 4) << 32)                  // stride byte offset: 8 rows x 128 B
         | ((uint64_t)1 << 46)                            // descriptor version
         | ((uint64_t)2 << 61);                           // 128-byte swizzle
}

// Instruction descriptor, kind::tf32: fp32 accumulator, TF32 A and B, both
// K-major, shape M x N.
__host__ __device__ constexpr uint32_t idesc_tf32(int m, int n)
{
    return (1u << 4)                                      // D format: F32
         | (2u << 7)                                      // A format: TF32
         | (2u << 10)                                     // B format: TF32
         | ((uint32_t)(n >> 3) << 17)                     // N / 8
         | ((uint32_t)(m >> 4) << 24);                    // M / 16
}

// Byte offset of element (row r, column c) of a K-major 128-byte-swizzled fp32
// tile with `rows` rows.
__host__ __device__ constexpr uint32_t sw128_offset(int r, int c, int rows)
{
    return (uint32_t)((c >> 5) * rows * 128 + r * 128 + ((((c & 31) >> 2) ^ (r & 7)) << 4) + ((c & 3) << 2));
}

// ---------------------------------------------------------------- tensor memory

// Allocate `ncols` columns (a power of two >= 32) by one whole warp; the base
// address is written to `*dst` in shared memory.
__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols)
{
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(dst);
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(s), "r"(ncols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Make this thread's generic-proxy shared-memory writes visible to the tensor core.
__device__ __forceinline__ void fence_smem_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// ---------------------------------------------------------------- MMA

// D[tmem] (+)= A[smem] * B[smem]^T  (both K-major), one K = 8 step.
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}"
                 ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]^T, one K = 8 step (A: lane = row, 8 columns).
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}"
                 ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}
// The mbarrier at `bar` gets one arrive once every MMA this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint64_t *bar)
{
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(bar);
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(s) : "memory");
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(bar);
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(s), "r"(count) : "memory");
}
// Wait for the phase with parity `parity` to complete, at most `limit` polls
// (each poll may suspend the thread for a while in hardware).  Returns false if
// the limit ran out.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint32_t limit)
{
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(bar);
    for (uint32_t i = 0; i < limit; ++i) {
        uint32_t done;
        asm volatile("{\n\t.reg .pred p;\n\t"
                     "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                     "selp.u32 %0, 1, 0, p;\n\t}"
                     : "=r"(done) : "r"(s), "r"(parity) : "memory");
        if (done) return true;
    }
    return false;
}

// ---------------------------------------------------------------- tensor memory <-> registers

// 32 consecutive 32-bit columns of this thread's lane (warp w reads lanes
// 32*(w%4) .. +31; taddr carries that lane base).  Call ld_wait() before use.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32])
{
    uint32_t r[32];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                   "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
                   "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
                   "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr) : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
                 "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
                 "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
                 ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
                   "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
                   "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
                   "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
                   "r"(r[29]), "r"(r[30]), "r"(r[31]) : "memory");
}
// 8 consecutive 32-bit columns of this thread's lane (as tmem_ld32).
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8])
{
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr) : "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
                 ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
                   "r"(r[7]) : "memory");
}
__device__ __forceinline__ void ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------- precision split

// x = hi + lo with hi the nearest TF32 value (low 13 mantissa bits zero, ties
// away from zero) and lo = x - hi, exact in fp32; the tensor core reads lo to
// TF32 precision (dropping at most 2^-10 of it, ~2^-21 of x), so a product of
// two split operands taken as hi*hi + hi*lo + lo*hi carries about 21
// significant bits (the lo*lo term, ~2^-22 relative, is dropped).  (Rounding lo
// to TF32 here as well measured the same error against the fp64 oracle, one
// instruction more per element.)  hi is rounded by integer arithmetic on the
// bits -- half of the dropped unit added to the magnitude, then the dropped
// bits cleared, which is that rounding for every finite x -- rather than by
// the conversion instruction, whose lower throughput cost the chunked prefill
// 4 % (2.370 -> 2.272 ms at batch 8, T 4096, bit for bit the same results).
__device__ __forceinline__ void split_tf32(float x, uint32_t &hi, uint32_t &lo)
{
    const uint32_t h = (__float_as_uint(x) + 0x1000u) & 0xFFFFE000u;
    hi = h;
    lo = __float_as_uint(x - __uint_as_float(h));
}

}  // namespace tc

// Launcher of the chunked tensor-core prefill (gdn_prefill_tc.cu): D == 128,
// k and q rows 16-byte aligned.  Needs the PrefillParams of gdn_internal.cuh.
struct PrefillParams;
cudaError_t launch_prefill_tc(const PrefillParams &p, bool f16_state, cudaStream_t s);
// Count of bounded MMA-completion waits that ran out on the current device.
cudaError_t tc_wait_timeouts(unsigned *count);
// Polls of an MMA completion before a tensor-core kernel launched after this call gives up.
void tc_set_wait_polls(uint32_t polls);
// The bound of the MMA waits alone (the tensor-copy waits keep theirs).
void tc_set_mma_wait_polls(uint32_t polls);

}  // namespace gdn
