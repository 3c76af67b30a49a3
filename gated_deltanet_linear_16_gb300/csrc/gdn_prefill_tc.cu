// gdn_prefill_tc.cu -- the prefill recurrence regrouped into chunks of 64
// tokens, with the chunk's matrix products on the fifth-generation tensor
// cores (tcgen05, TF32 operands split in two for fp32-level accuracy).
//
// The recurrence is the one of logicaffeine_compile/codegen_cuda/gdn.rs,
// kernel `gdn_step`, applied token by token as
// metrale_model_layers/layers/ops/ssm_gdn_a.rs, `gdn_prefill_regresident`,
// does: S_t = alpha_t S_{t-1} + delta_t k_t^T with
// delta_t = beta_t (v_t - alpha_t S_{t-1} k_t), o_t = S_t q_t / sqrt(D).
// Unrolled over a chunk of C tokens from the state S at its start (gamma_t =
// alpha_0 ... alpha_t with t counted from 0 in the chunk, rho(t,i) = alpha_{i+1}
// ... alpha_t, taken as a product, never as the ratio gamma_t / gamma_i):
//
//   S_t   = gamma_t S + sum_{i<=t} rho(t,i) delta_i k_i^T
//   delta_t + beta_t sum_{i<t} rho(t,i) (k_t.k_i) delta_i = beta_t (v_t - gamma_t S k_t)
//   o_t   = (gamma_t S q_t + sum_{i<=t} rho(t,i) (q_t.k_i) delta_i) / sqrt(D)
//
// i.e. (I + A) Delta = R with A[t][i] = beta_t rho(t,i) k_t.k_i (i < t), so
// Delta = T R with T = (I + A)^-1 (unit lower triangular), and at the chunk's
// end S <- gamma_C S + Delta^T Ktilde with Ktilde[t] = rho(C,t) k_t.  This is
// the same arithmetic in real numbers (the chunked "WY" form of the delta
// rule); only the fp32 rounding differs.  Per chunk and head, in order:
//
//   SIMT   the state, split, into TMEM; the low parts of the chunk's [K;Q] tile
//          (the tile itself arrived by tensor copies) into shared memory: half of
//          them already written while the previous chunk's MMA-3 ran
//   MMA-1  G = [K;Q] K^T (128 x 64, two issuers over the halves of K) and
//          Y = S [K;Q]^T (128 x 128, S from TMEM, one issuer)
//   SIMT   gamma, rho(C,.) by warp scans; A from G (warps 0, 1, 4, 5, while Y
//          runs); T = (I + A)^-1 (16 x 16 diagonal blocks, then block
//          products); P from G; R^T = beta (v - gamma Y_K) into TMEM; T, P,
//          Ktilde^T into shared memory
//   MMA-2  Delta^T = R^T T^T (128 x 64, one issuer and accumulator per pass)
//   SIMT   Delta^T = sum of the passes, split into TMEM
//   MMA-3  [Z | (P Delta)^T] = Delta^T [Ktilde | P^T] (128 x 192, two issuers
//          over the halves of K)
//   SIMT   o_t = (gamma_t Y_Q + P Delta) / sqrt(D) into a shared-memory tile
//          written out by one tensor store;  S <- gamma_C S + Z (fp32)
//
// Every MMA operand x is split as x = hi + lo with hi the nearest TF32 value and
// lo = x - hi (read as TF32 by the tensor core), and a product is taken as
// hi*hi + hi*lo + lo*hi (three passes), which carries about 21 significant bits
// per product; k and q take hi = x truncated to TF32 instead (about 19 bits
// per product: their copies arrive in the operand layout, so only lo is
// computed); the accumulators are fp32 in tensor memory.  The exact fp32
// state stays in registers (thread = row a of the head, half of its columns);
// only its split copy is in tensor memory.
//
// One CTA (8 warps) per (sequence, value head); warp w owns tensor-memory lanes
// 32*(w%4).. (rows of the state) and half w/4 of the columns it loads.  Lane 0
// of warps 2, 3 and 6 issue the MMAs (one thread issues one MMA per ~120-140
// cycles whatever its N, and MMAs from several threads proceed together), so
// each product is split over two or three issuers, each part into its own
// accumulator (tensor memory, all 512 columns in use during MMA-1, keeps Y on
// one issuer).  The next chunk's k and q arrive during the current chunk by
// eight TMA tensor copies straight into the 128-byte-swizzled operand layout
// (their fp32 bits serve as the high TF32 parts: the tensor core reads the top
// 19 bits, and only the exact low parts x - trunc(x) are computed), alpha and
// beta by cp.async; the chunk's outputs leave by one tensor store (TMA) of a
// 32 KB tile.  Both keep per-lane global accesses out of the load/store queue
// that the chunk's shared-memory work needs (2.82 -> 2.46 ms at batch 8, T
// 4096); v keeps plain loads (in shared memory its reads cost wavefronts of
// the pipe the SIMT phases are bound by).  The CTA holds all 512 tensor-memory
// columns and ~230 KB of shared memory, so an SM runs one such CTA at a time.
// Loops stay rolled where they can: the chunk body runs once per chunk, so
// instruction fetch is a cost.  The only waits are on the CTA's own MMA and
// tensor-copy completions (mbarriers armed by tcgen05.commit or by the
// copies' transaction counts), each bounded: if a bound ran out (or was set to
// 0 to test this path), the CTA stops, lets the MMAs and copies it issued
// finish (again bounded), counts the event in g_tc_wait_timeouts and writes NaN
// to its state.
#include <atomic>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "gdn_internal.cuh"
#include "gdn_tc.cuh"

__device__ unsigned int g_tc_wait_timeouts;

namespace gdn {
namespace {

constexpr int kD = 128;
constexpr int kC = 64;                       // tokens per chunk
constexpr int kThreads = 256;
// MMA-issuing threads: lane 0 of warps 2, 3 and 6 (no part in building A).  One thread issues about
// one MMA per ~120-140 cycles whatever its N, while the tensor core takes MMAs from several threads
// at once, so each product is split over up to three issuers, each part (a range of K, or a pass of
// the precision split) into its own accumulator, summed by the SIMT phase after.
constexpr int kIss0 = 64, kIss1 = 96, kIss2 = 192;
constexpr uint32_t kWaitLimit = 1u << 22;    // polls of an mbarrier phase before giving up

// shared memory (1024-aligned), byte offsets
// [K;Q]: 128 rows x 128, until MMA-1 and the k reads are done.  kKQHi: as the tensor copies bring it
// in (during the previous chunk), its fp32 bits the high TF32 parts (the tensor core reads the top 19
// bits); kKQLo: the low parts x - trunc_tf32(x), exact.  T and the B operand of MMA-3 reuse
// [0, 128 KB) after MMA-1; the next chunk's copies land in kKQHi once the k reads are done, and
// the low parts of its k-blocks 0-1 go into T's 32 KB while MMA-3 runs.
constexpr uint32_t kKQLo = 0, kKQHi = 131072;
constexpr uint32_t kTHi = 0, kTLo = 16384;             // T: 64 rows (t) x 64 (i), after MMA-1
// B operand of MMA-3, 192 rows x 64 (K = t or i): rows 0-127 Ktilde^T (row c), rows 128-191 P (row t)
constexpr uint32_t kBHi = 32768, kBLo = 81920;
constexpr int kBRows = 192;
// fp32 64 x 64 work matrix W (row stride kAS): A in its strict lower triangle, T = (I + A)^-1
// transposed in its upper triangle and diagonal (T[t][j] at W[j][t]); then a 32 x 36 scratch Xs and
// Tr, T's top-left 32 x 32 block row-major (zeros above the diagonal), both with 16-byte rows so the
// 32 x 32 block product reads four consecutive columns in one load
constexpr int kAS = 65, kXS = 36, kTS = 36;
constexpr uint32_t kWOff = kKQHi + 65536, kXsOff = kWOff + kC * kAS * 4, kTrOff = kXsOff + 32 * kXS * 4;
// the chunk's outputs o[t][a] (64 x 128 fp32, row-major) for one tensor store, over W and the scratch
// after them: written in the last phase, read out by the copy engine before the next chunk builds A
constexpr uint32_t kOStage = kWOff, kOBytes = kC * kD * 4;
constexpr uint32_t kSmemEnd = (kTrOff + 32 * kTS * 4 > kOStage + kOBytes) ? kTrOff + 32 * kTS * 4 : kOStage + kOBytes;
constexpr uint32_t kSmemBytes = kSmemEnd + 1024;                        // + alignment slack

// tensor-memory columns
constexpr uint32_t kSHi = 0, kSLo = 128;     // split state (A operand of Y)
constexpr uint32_t kY = 256, kYQ = 320;      // Y = S [K;Q]^T: columns t of K, then of Q (all three passes)
constexpr uint32_t kG = 384, kGb = 448;      // G = [K;Q] K^T over the first and the second half of K
constexpr uint32_t kRHi = 384, kRLo = 448;   // split R^T (after G is read)
constexpr uint32_t kD1 = 128, kD2 = 0, kD3 = 64;   // Delta^T = R^T T^T, one accumulator per pass (after Y)
constexpr uint32_t kDtHi = 192, kDtLo = 256; // split Delta^T
// Delta^T [Ktilde | P^T] (N = 192) over the first and the second half of K (t) at kM3a and kM3b;
// Z in the first 128 columns of each, (P Delta)^T in the last 64
constexpr uint32_t kM3a = 0, kM3b = 320;

struct __align__(16) ChunkScalars {
    float gamma[kC];          // gamma_t = alpha_0 ... alpha_t (chunk-local, t from 0)
    float rho_last[kC];       // rho(C-1, t) = alpha_{t+1} ... alpha_{C-1}
    float sigma[kC];          // sigma_i = alpha_32 ... alpha_i for i >= 32 (= rho(i, 31))
};

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ void st_shared_b32(uint32_t addr, uint32_t a)
{
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(a) : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}
__device__ __forceinline__ float ld_shared_f32(uint32_t addr)
{
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ void cp_async4_s(uint32_t saddr, const void *gmem)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(saddr), "l"(gmem) : "memory");
}
// Four split values stored as 16-byte hi and lo vectors.
__device__ __forceinline__ void st_split4(uint32_t hi_addr, uint32_t lo_addr, float a, float b, float c, float d)
{
    uint32_t h0, h1, h2, h3, l0, l1, l2, l3;
    tc::split_tf32(a, h0, l0); tc::split_tf32(b, h1, l1);
    tc::split_tf32(c, h2, l2); tc::split_tf32(d, h3, l3);
    st_shared_v4(hi_addr, h0, h1, h2, h3);
    st_shared_v4(lo_addr, l0, l1, l2, l3);
}

// Passes [p0, p1) of the split product over the K/8 steps [k0, k1): pass 0 = A_hi B_hi, 1 = A_hi
// B_lo, 2 = A_lo B_hi, all into D (the first MMA overwrites it).  A in shared memory (a_hi/a_lo
// descriptors' base addresses) or tensor memory.  Issued by one thread.  The loops stay rolled:
// this kernel's code is run once per chunk by few warps, so its size (instruction fetch) matters
// more than the loop overhead.
template <bool A_TMEM>
__device__ __forceinline__ void mma_passes(uint32_t d, uint32_t a_hi, uint32_t a_lo, uint32_t b_hi, uint32_t b_lo,
                                           uint32_t a_block, uint32_t b_block, int k0, int k1, uint32_t idesc,
                                           int p0, int p1)
{
#pragma unroll 1
    for (int pass = p0; pass < p1; ++pass) {
        const uint32_t a = pass == 2 ? a_lo : a_hi;
        const uint32_t b = pass == 1 ? b_lo : b_hi;
#pragma unroll 1
        for (int kk = k0; kk < k1; ++kk) {
            const uint32_t acc = (pass > p0 || kk > k0) ? 1u : 0u;
            const uint64_t bd = tc::smem_desc_sw128(b + (kk >> 2) * b_block + (kk & 3) * 32);
            if constexpr (A_TMEM) {
                tc::mma_ts(d, a + kk * 8, bd, idesc, acc);
            } else {
                tc::mma_ss(d, tc::smem_desc_sw128(a + (kk >> 2) * a_block + (kk & 3) * 32), bd, idesc, acc);
            }
        }
    }
}

// Every thread: tensor-core ops and shared-memory writes so far are visible to
// the MMA-issuing thread after this.
__device__ __forceinline__ void sync_for_mma()
{
    tc::fence_smem_async();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
}
// AND of `pred` over the 128 threads of warps 0, 1, 4, 5 (named barrier 1).
__device__ __forceinline__ bool and_a_warps(bool pred)
{
    uint32_t r;
    asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
                 "bar.red.and.pred q, 1, 128, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
                 : "=r"(r) : "r"((uint32_t)pred) : "memory");
    return r != 0;
}

// Chunk [c0, c0 + 64) of k and q by eight tensor copies (one per 32-column block of each: 64 tokens x
// 128 bytes with the 128-byte swizzle, the layout the MMAs read) into the [K;Q] tile at `dst`; tokens
// past the sequence's end read as zeros.  They complete on `bar`, whose transaction count (64 KB) is
// armed here.  One thread.
__device__ __forceinline__ void load_kq(const CUtensorMap *kmap, const CUtensorMap *qmap, uint32_t dst, uint64_t *bar,
                                        int g, int c0, int seq)
{
    const uint32_t b = (uint32_t)__cvta_generic_to_shared(bar);
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(b), "r"(65536u) : "memory");
#pragma unroll
    for (int kb = 0; kb < 4; ++kb) {
#pragma unroll
        for (int m = 0; m < 2; ++m)
            asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
                         " [%0], [%1, {%2, %3, %4}], [%5];"
                         ::"r"(dst + kb * 16384 + m * 8192), "l"(m == 0 ? kmap : qmap), "r"(g * kD + kb * 32),
                           "r"(c0), "r"(seq), "r"(b) : "memory");
    }
}

// alpha, beta of chunk [c0, c0 + n) into ab[0], ab[1] with cp.async (threads 0-63); padding tokens get
// alpha = 1, beta = 0.  Each copier waits for its own copies before the barrier that publishes them.
__device__ __forceinline__ void prefetch_ab(float (*ab)[kC], const PrefillParams &p, int seq, int h, int c0, int n,
                                            int tid)
{
    if (tid < kC) {
        const uint32_t sa = (uint32_t)__cvta_generic_to_shared(&ab[0][tid]);
        const uint32_t sb = (uint32_t)__cvta_generic_to_shared(&ab[1][tid]);
        if (tid < n) {
            const int64_t row = (int64_t)seq * p.seq_len + c0 + tid;
            cp_async4_s(sa, p.alpha + row * p.gb_stride + h);
            cp_async4_s(sb, p.beta + row * p.gb_stride + h);
        } else {
            st_shared_b32(sa, __float_as_uint(1.0f));
            st_shared_b32(sb, 0u);
        }
    }
    cp_async_commit();
}

// The low TF32 part of x: x minus its top 19 bits (exact).
__device__ __forceinline__ uint32_t tf32_low(uint32_t x)
{
    return __float_as_uint(__uint_as_float(x) - __uint_as_float(x & 0xFFFFE000u));
}

// The chunk's o tile (shared memory, row-major [t][a]) to o[seq][c0 + t][h D + a] by one tensor store
// through a 3-D map (columns, tokens, sequences): rows past the sequence's end fall outside the map and
// are not written.  Issued by one thread after every thread's shared-memory writes were made visible to
// the copy engine (fence.proxy.async) and a barrier.
__device__ __forceinline__ void store_o_tile(const CUtensorMap *map, uint32_t src, int x, int y, int z)
{
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];"
                 ::"l"(map), "r"(x), "r"(y), "r"(z), "r"(src) : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until the copy engine has read the tile out of shared memory (the buffer may be written again).
__device__ __forceinline__ void o_tile_read_done() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Wait until the stores are complete.
__device__ __forceinline__ void o_tile_done() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Barrier among the 128 threads of warps 0, 1, 4 and 5 (named barrier 1).
__device__ __forceinline__ void sync_a_warps() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// T = (I + A)^-1 for the strictly lower triangular 64 x 64 A in W (row stride
// kAS); T[t][j] (t >= j) is written to W[j][t], the upper triangle and the
// diagonal, which A leaves free.  First the four 16 x 16 diagonal blocks by
// forward substitution (64 threads, one per column: invert_diag_blocks), then
// the blocks under the diagonal from [[M11, 0], [M21, M22]]^-1 = [[T11, 0],
// [-T22 M21 T11, T22]]: the two 16 x 16 ones by the 128 threads that built A
// (invert_off_diag16, before Y's issuing warp is free), then the 32 x 32 one by
// four warps (invert_off_diag32).  Xs: 32 x 36 scratch; Tr: row-major copy of T[0..31][0..31].
__device__ __forceinline__ float w_a(const float *W, int t, int i) { return W[t * kAS + i]; }
__device__ __forceinline__ float &w_t(float *W, int t, int j) { return W[j * kAS + t]; }

__device__ __forceinline__ void invert_diag_blocks(float *W, float *Tr, int it)
{
    const int kb = it >> 4, jj = it & 15, base = 16 * kb;
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = i == jj ? 1.0f : 0.0f;
#pragma unroll
    for (int t = 1; t < 16; ++t) {
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int i = 0; i + 1 < t; i += 2) {
            a0 = fmaf(w_a(W, base + t, base + i), x[i], a0);
            a1 = fmaf(w_a(W, base + t, base + i + 1), x[i + 1], a1);
        }
        if (t & 1) a0 = fmaf(w_a(W, base + t, base + t - 1), x[t - 1], a0);
        if (t > jj) x[t] = -(a0 + a1);
    }
#pragma unroll
    for (int t = 0; t < 16; ++t)
        if (t >= jj) w_t(W, base + t, base + jj) = x[t];
    if (kb < 2) {                                  // Tr: this column of the block (x[t] = 0 above it)
#pragma unroll
        for (int t = 0; t < 16; ++t) Tr[(base + t) * kTS + base + jj] = x[t];
        if (kb == 0) {                             // and the zero block right of it
#pragma unroll
            for (int t = 0; t < 16; ++t) Tr[t * kTS + 16 + jj] = 0.0f;
        }
    }
}

// The two 16 x 16 blocks by the 128 threads of warps 0, 1, 4, 5 (it = 0..127, four outputs each).
__device__ __forceinline__ void invert_off_diag16(float *W, float *Xs, float *Tr, int it)
{
    {   // X = M21 T11 for the pairs (rows 16..31, cols 0..15) and (rows 48..63, cols 32..47): row t, cols j0..+3
        const int b = it >> 6, t = (it >> 2) & 15, j0 = 4 * (it & 3), base = 32 * b;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float a = w_a(W, base + 16 + t, base + i);
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[e] = fmaf(a, i >= j0 + e ? w_t(W, base + i, base + j0 + e) : 0.0f, acc[e]);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) Xs[(16 * b + t) * kXS + j0 + e] = acc[e];
    }
    sync_a_warps();
    {   // T21 = -T22 X for the two pairs
        const int b = it >> 6, t = (it >> 2) & 15, j0 = 4 * (it & 3), base = 32 * b;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float tv = i <= t ? w_t(W, base + 16 + t, base + 16 + i) : 0.0f;
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[e] = fmaf(tv, Xs[(16 * b + i) * kXS + j0 + e], acc[e]);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) w_t(W, base + 16 + t, base + j0 + e) = -acc[e];
        if (b == 0) {                              // the block under T's first diagonal block, into Tr
#pragma unroll
            for (int e = 0; e < 4; ++e) Tr[(16 + t) * kTS + j0 + e] = -acc[e];
        }
    }
}

// The 32 x 32 block by the 128 threads of warps 0-3 (named barrier 2), a 2 x 4 block of outputs each
// (rows 2 ti, 2 ti + 1, columns 4 tj .. +3): per step along the inner dimension two scalar loads and
// one 16-byte load feed 8 FMAs.  Shared-memory wavefronts bound this product (a 16-byte load costs
// four), so larger blocks on fewer warps beat four outputs on all eight.  T11 from Tr, X through Xs.
__device__ __forceinline__ void invert_off_diag32(float *W, float *Xs, const float *Tr, int tid)
{
    const int ti = tid >> 3, tj = tid & 7, t0 = 2 * ti, j0 = 4 * tj;
    {   // X = M21 T11: rows t0, t0+1, cols j0 .. j0+3
        float4 acc[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
        for (int i = 0; i < 32; ++i) {
            const float4 tr = *reinterpret_cast<const float4 *>(Tr + i * kTS + j0);
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const float a = w_a(W, 32 + t0 + k, i);
                acc[k].x = fmaf(a, tr.x, acc[k].x);
                acc[k].y = fmaf(a, tr.y, acc[k].y);
                acc[k].z = fmaf(a, tr.z, acc[k].z);
                acc[k].w = fmaf(a, tr.w, acc[k].w);
            }
        }
#pragma unroll
        for (int k = 0; k < 2; ++k) *reinterpret_cast<float4 *>(Xs + (t0 + k) * kXS + j0) = acc[k];
    }
    asm volatile("bar.sync 2, 128;" ::: "memory");
    {   // T21 = -T22 X (T22 lower triangular: zero for i > t)
        float4 acc[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
        for (int i = 0; i < 32; ++i) {
            const float4 x = *reinterpret_cast<const float4 *>(Xs + i * kXS + j0);
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const float tv = i <= t0 + k ? w_t(W, 32 + t0 + k, 32 + i) : 0.0f;
                acc[k].x = fmaf(tv, x.x, acc[k].x);
                acc[k].y = fmaf(tv, x.y, acc[k].y);
                acc[k].z = fmaf(tv, x.z, acc[k].z);
                acc[k].w = fmaf(tv, x.w, acc[k].w);
            }
        }
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            w_t(W, 32 + t0 + k, j0) = -acc[k].x;
            w_t(W, 32 + t0 + k, j0 + 1) = -acc[k].y;
            w_t(W, 32 + t0 + k, j0 + 2) = -acc[k].z;
            w_t(W, 32 + t0 + k, j0 + 3) = -acc[k].w;
        }
    }
}

template <typename TS, bool TMA_O>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_d128(const PrefillParams p, const uint32_t polls, const uint32_t copy_polls,
                const __grid_constant__ CUtensorMap o_map,
                const __grid_constant__ CUtensorMap k_map, const __grid_constant__ CUtensorMap q_map)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    float *W = reinterpret_cast<float *>(smem + kWOff);
    float *Xs = reinterpret_cast<float *>(smem + kXsOff);
    float *Tr = reinterpret_cast<float *>(smem + kTrOff);
    __shared__ ChunkScalars sc;
    __shared__ __align__(16) float ab[2][2][kC];    // [chunk parity][alpha, beta][t]
    __shared__ uint64_t bars[5];                    // G (2 issuers), Y (1), MMA-2 (3), MMA-3 (2), [K;Q] copies
    __shared__ uint32_t tmem_base;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, hf = warp >> 2;
    const int r = 32 * quad + lane;                 // tensor-memory lane = state row a = token row
    const uint32_t lanebase = (uint32_t)(32 * quad) << 16;
    const int head = blockIdx.x;
    const int seq = head / p.nv;
    const int h = head - seq * p.nv;
    const int g = h % p.nk;
    const int T = p.seq_len;
    const uint32_t sbase = (uint32_t)__cvta_generic_to_shared(smem);

    const float *vbase = p.v + (int64_t)seq * T * p.v_stride + (int64_t)h * kD;
    float *obase = p.o + (int64_t)seq * T * p.o_stride + (int64_t)h * kD;

    prefetch_ab(ab[0], p, seq, h, 0, min(kC, T), tid);
    if (warp == 0) tc::tmem_alloc(&tmem_base, 512);
    if (tid == 0) {
        tc::mbar_init(&bars[0], 2);
        tc::mbar_init(&bars[1], 1);
        tc::mbar_init(&bars[2], 3);
        tc::mbar_init(&bars[3], 2);
        tc::mbar_init(&bars[4], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (tid == 0) load_kq(&k_map, &q_map, sbase + kKQHi, &bars[4], g, 0, seq);
    uint32_t kq_ph = 0;                             // parity of the [K;Q] copies' phase being awaited
    bool kq_pend = true;                            // copies in flight not yet seen complete
    const uint32_t tm = tmem_base + lanebase;       // this warp's lanes
    uint32_t ph = 0;                                // parity of this chunk's phase of each barrier

    // the exact state: row r, columns 64*hf .. +63, in registers
    TS *srow = reinterpret_cast<TS *>(p.state) + seq * p.pitch + (int64_t)h * kD * kD + (int64_t)r * kD + 64 * hf;
    float S[64];
#pragma unroll
    for (int j = 0; j < 64; ++j) S[j] = to_f32<TS>(srow[j]);
    bool ok = true;
    bool lo_half = false;                           // k-blocks 0-1 of this chunk's low parts already done
    uint32_t pend = 0;                              // barriers with a committed phase not yet seen complete

    for (int c0 = 0, par = 0; c0 < T && ok; c0 += kC, par ^= 1) {
        const int n = min(kC, T - c0);
        const float *alpha = ab[par][0], *beta = ab[par][1];
        // ---- 0. the state, split, into tensor memory (A operand of Y) ----
#pragma unroll
        for (int cb = 0; cb < 2; ++cb) {
            uint32_t hi[32], lo[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) tc::split_tf32(S[32 * cb + j], hi[j], lo[j]);
            tc::tmem_st32(tm + kSHi + 64 * hf + 32 * cb, hi);
            tc::tmem_st32(tm + kSLo + 64 * hf + 32 * cb, lo);
        }
        // ---- 1. the low parts of the [K;Q] tile (the tensor copies brought the high parts) ----
        const bool okk = tc::mbar_wait(&bars[4], kq_ph, copy_polls);
        cp_async_wait<0>();                                // this thread's alpha, beta copies
        if (lo_half) {                 // k-blocks 0-1 were done during the previous chunk's MMA-3
#pragma unroll 2
            for (int i = 0; i < 8; ++i) {
                const uint32_t off = tc::sw128_offset(16 * warp + 2 * i + (lane >> 4), 64 + 4 * (lane & 15), 128);
                const uint4 x = ld_shared_v4(sbase + kKQHi + off);
                st_shared_v4(sbase + kKQLo + off, tf32_low(x.x), tf32_low(x.y), tf32_low(x.z), tf32_low(x.w));
            }
        } else {
#pragma unroll 2
            for (int i = 0; i < 16; ++i) {
                const uint32_t off = tc::sw128_offset(16 * warp + i, 4 * lane, 128);
                const uint4 x = ld_shared_v4(sbase + kKQHi + off);
                st_shared_v4(sbase + kKQLo + off, tf32_low(x.x), tf32_low(x.y), tf32_low(x.z), tf32_low(x.w));
            }
        }
        tc::st_wait();                                     // the split state is in tensor memory
        if (TMA_O && tid == 0) o_tile_read_done();        // the last chunk's o tile is out of W's space
        // ---- MMA-1: G = [K;Q] K^T (two issuers, bars[0]) and Y = S [K;Q]^T (one issuer, bars[1]) ----
        tc::fence_smem_async();
        tc::fence_before_sync();
        ok = __syncthreads_and(okk) != 0;                  // [K;Q] and alpha, beta complete
        tc::fence_after_sync();
        if (!ok) break;
        kq_pend = false;
        kq_ph ^= 1u;
        if (tid == kIss0 || tid == kIss2) {       // G over the first / second half of K
            const bool first = tid == kIss0;
            mma_passes<false>(tmem_base + (first ? kG : kGb), sbase + kKQHi, sbase + kKQLo, sbase + kKQHi,
                              sbase + kKQLo, 128 * 128, 128 * 128, first ? 0 : kD / 16, first ? kD / 16 : kD / 8,
                              tc::idesc_tf32(128, 64), 0, 3);
            tc::mma_commit(&bars[0]);
        } else if (tid == kIss1) {
            mma_passes<true>(tmem_base + kY, tmem_base + kSHi, tmem_base + kSLo, sbase + kKQHi, sbase + kKQLo,
                             0, 128 * 128, 0, kD / 8, tc::idesc_tf32(128, 128), 0, 3);
            tc::mma_commit(&bars[1]);
        }
        __syncwarp();
        pend = 0x3u;
        // products of the decays, by warps that build A (they wait for G next): gamma (prefix),
        // rho(C-1, .) (suffix), sigma (prefix from 32); published by the A warps' barrier and the full
        // barriers after
        if (warp == 0 || warp == 1 || warp == 5) {
            if (warp == 5) {
                float pr = alpha[32 + lane];
#pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    const float y = __shfl_up_sync(kFull, pr, d);
                    if (lane >= d) pr = y * pr;
                }
                sc.sigma[32 + lane] = pr;
            } else {
                const float a0 = alpha[2 * lane], a1 = alpha[2 * lane + 1];
                float pr = a0 * a1;
                if (warp == 0) {
#pragma unroll
                    for (int d = 1; d < 32; d <<= 1) {
                        const float y = __shfl_up_sync(kFull, pr, d);
                        if (lane >= d) pr = y * pr;
                    }
                    float ex = __shfl_up_sync(kFull, pr, 1);
                    if (lane == 0) ex = 1.0f;
                    const float g0 = ex * a0;
                    sc.gamma[2 * lane] = g0;
                    sc.gamma[2 * lane + 1] = g0 * a1;
                } else {
#pragma unroll
                    for (int d = 1; d < 32; d <<= 1) {
                        const float y = __shfl_down_sync(kFull, pr, d);
                        if (lane + d < 32) pr = y * pr;
                    }
                    float ex = __shfl_down_sync(kFull, pr, 1);
                    if (lane == 31) ex = 1.0f;
                    sc.rho_last[2 * lane + 1] = ex;
                    sc.rho_last[2 * lane] = a1 * ex;
                }
            }
        }

        // the next chunk's alpha, beta on their way while this one is computed (k and q follow once
        // MMA-1 and the k reads below are done with the tile)
        if (c0 + kC < T) prefetch_ab(ab[par ^ 1], p, seq, h, c0 + kC, min(kC, T - c0 - kC), tid);
        // v_t[a] for t = 32 hf + j, a = r (coalesced across the warp's lanes)
        float vv[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const int t = 32 * hf + j;
            vv[j] = t < n ? __ldg(vbase + (int64_t)(c0 + t) * p.v_stride + r) : 0.0f;
        }
        // ---- 2. A from G by warps 0, 1, 4, 5 (lanes 0-63), the diagonal blocks of T = (I + A)^-1 by
        //         warps 0 and 1, the rest of T by all warps, while Y is still on the tensor core ----
        bool ok_g = true;
        if (r < kC) {
            ok_g = and_a_warps(tc::mbar_wait(&bars[0], ph, polls));
            tc::fence_after_sync();
            // A[t][i] = beta_t rho(t,i) k_t.k_i, t = r, i = 32 hf + 8 grp + e, walked downwards (G is
            // read only once it is known complete: after a timeout, A stays as it was)
            const int t = r;
            float pr = (hf == 0 && t >= 32) ? sc.sigma[t] : 1.0f;
            const float bt = beta[t];
#pragma unroll 1
            for (int grp = ok_g ? 3 : -1; grp >= 0; --grp) {
                float gv[8], gw[8];
                tc::tmem_ld8(tm + kG + 32 * hf + 8 * grp, gv);
                tc::tmem_ld8(tm + kGb + 32 * hf + 8 * grp, gw);
                const float4 a_lo = *reinterpret_cast<const float4 *>(alpha + 32 * hf + 8 * grp);
                const float4 a_hi = *reinterpret_cast<const float4 *>(alpha + 32 * hf + 8 * grp + 4);
                const float al[8] = {a_lo.x, a_lo.y, a_lo.z, a_lo.w, a_hi.x, a_hi.y, a_hi.z, a_hi.w};
                tc::ld_wait();
#pragma unroll
                for (int e = 7; e >= 0; --e) {
                    const int i = 32 * hf + 8 * grp + e;
                    if (i < t) W[t * kAS + i] = bt * pr * (gv[e] + gw[e]);
                    if (i <= t) pr *= al[e];
                }
            }
            sync_a_warps();                                // A complete
            if (hf == 0) invert_diag_blocks(W, Tr, (warp & 1) * 32 + lane);
            sync_a_warps();                                // diagonal blocks of T done
            invert_off_diag16(W, Xs, Tr, (warp & 1) * 32 + lane + 64 * hf);
            tc::fence_before_sync();
        }
        __syncthreads();                                   // 16 x 16 blocks done; Y's issuer done issuing
        if (warp < 4) invert_off_diag32(W, Xs, Tr, tid);
        ok = __syncthreads_and(ok_g && tc::mbar_wait(&bars[1], ph, polls)) != 0;         // T complete, Y done
        tc::fence_after_sync();
        if (!ok) break;
        pend = 0;
        // k_t[c] (exact: the copied fp32 value) from the tile before the next chunk's copies overwrite it;
        // t = 32 hf + j, c = r
        float kv[32];
        {   // element (row 32 hf + j, column r) of the 128-row K-major tile: a row step is 128 bytes and
            // the 16-byte chunk is XOR-ed with the row's low three bits
            const uint32_t base = sbase + kKQHi + (r >> 5) * 128 * 128 + 32 * hf * 128 + ((r & 3) << 2);
            const uint32_t chunk = (r & 31) >> 2;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const uint32_t a = base + j * 128 + ((chunk ^ (uint32_t)(j & 7)) << 4);
                kv[j] = ld_shared_f32(a);                  // the copied fp32 value itself
            }
        }
        __syncthreads();
        if (c0 + kC < T) {                                 // MMA-1 and the k reads are done with the tile
            if (tid == 0) load_kq(&k_map, &q_map, sbase + kKQHi, &bars[4], g, c0 + kC, seq);
            kq_pend = true;
        }

        // ---- 2b. operands of MMA-2 and MMA-3: T, P, Ktilde^T to shared memory, R^T to tensor memory ----
        {   // T: row t = tid / 4, columns 16 (tid % 4) .. +15 (zero above the diagonal)
            const int t = tid >> 2, cb = (tid & 3) * 16;
#pragma unroll 1
            for (int jc = 0; jc < 4; ++jc) {
                const int c = cb + 4 * jc;
                const uint32_t off = tc::sw128_offset(t, c, kC);
                st_split4(sbase + kTHi + off, sbase + kTLo + off,
                          c <= t ? W[c * kAS + t] : 0.0f, c + 1 <= t ? W[(c + 1) * kAS + t] : 0.0f,
                          c + 2 <= t ? W[(c + 2) * kAS + t] : 0.0f, c + 3 <= t ? W[(c + 3) * kAS + t] : 0.0f);
            }
        }
        if (r >= kC) {    // P[t][i] = rho(t,i) q_t.k_i from G row 64 + t, i = 32 hf + 8 grp + e (zero for i > t)
            const int t = r - kC;
            float pr = (hf == 0 && t >= 32) ? sc.sigma[t] : 1.0f;
#pragma unroll 1
            for (int grp = 3; grp >= 0; --grp) {
                float gv[8], gw[8];
                tc::tmem_ld8(tm + kG + 32 * hf + 8 * grp, gv);
                tc::tmem_ld8(tm + kGb + 32 * hf + 8 * grp, gw);
                const float4 a_lo = *reinterpret_cast<const float4 *>(alpha + 32 * hf + 8 * grp);
                const float4 a_hi = *reinterpret_cast<const float4 *>(alpha + 32 * hf + 8 * grp + 4);
                const float al[8] = {a_lo.x, a_lo.y, a_lo.z, a_lo.w, a_hi.x, a_hi.y, a_hi.z, a_hi.w};
                tc::ld_wait();
#pragma unroll
                for (int e = 7; e >= 0; --e) {
                    const int i = 32 * hf + 8 * grp + e;
                    gv[e] = i <= t ? pr * (gv[e] + gw[e]) : 0.0f;
                    if (i <= t) pr *= al[e];
                }
                const uint32_t off = tc::sw128_offset(128 + t, 32 * hf + 8 * grp, kBRows);
                st_split4(sbase + kBHi + off, sbase + kBLo + off, gv[0], gv[1], gv[2], gv[3]);
                const uint32_t off2 = tc::sw128_offset(128 + t, 32 * hf + 8 * grp + 4, kBRows);
                st_split4(sbase + kBHi + off2, sbase + kBLo + off2, gv[4], gv[5], gv[6], gv[7]);
            }
        }
        {   // Ktilde^T[c][t] = rho(C-1, t) k_t[c]: row c = r, columns t = 32 hf + j (one K block)
#pragma unroll
            for (int jc = 0; jc < 8; ++jc) {
                const float4 rl = *reinterpret_cast<const float4 *>(sc.rho_last + 32 * hf + 4 * jc);
                const uint32_t off = tc::sw128_offset(r, 32 * hf + 4 * jc, kBRows);
                st_split4(sbase + kBHi + off, sbase + kBLo + off, rl.x * kv[4 * jc], rl.y * kv[4 * jc + 1],
                          rl.z * kv[4 * jc + 2], rl.w * kv[4 * jc + 3]);
            }
        }
        {   // R^T[a][t] = beta_t (v_t[a] - gamma_t Y_K[a][t]), t = 32 hf + j, over G's columns (each
            // warp writes only the columns it alone read, or that no warp reads)
            float yk[32];
            tc::tmem_ld32(tm + kY + 32 * hf, yk);
            tc::ld_wait();
            uint32_t rhi[32], rlo[32];
#pragma unroll
            for (int jc = 0; jc < 8; ++jc) {
                const float4 bt = *reinterpret_cast<const float4 *>(beta + 32 * hf + 4 * jc);
                const float4 gm = *reinterpret_cast<const float4 *>(sc.gamma + 32 * hf + 4 * jc);
                const int j = 4 * jc;
                tc::split_tf32(bt.x * (vv[j] - gm.x * yk[j]), rhi[j], rlo[j]);
                tc::split_tf32(bt.y * (vv[j + 1] - gm.y * yk[j + 1]), rhi[j + 1], rlo[j + 1]);
                tc::split_tf32(bt.z * (vv[j + 2] - gm.z * yk[j + 2]), rhi[j + 2], rlo[j + 2]);
                tc::split_tf32(bt.w * (vv[j + 3] - gm.w * yk[j + 3]), rhi[j + 3], rlo[j + 3]);
            }
            tc::tmem_st32(tm + kRHi + 32 * hf, rhi);
            tc::tmem_st32(tm + kRLo + 32 * hf, rlo);
            tc::st_wait();
        }

        // ---- MMA-2: Delta^T = R^T T^T, one pass per issuer and accumulator ----
        sync_for_mma();
        if (tid == kIss0 || tid == kIss1 || tid == kIss2) {
            const int pass = tid == kIss0 ? 0 : (tid == kIss1 ? 1 : 2);
            mma_passes<true>(tmem_base + (pass == 0 ? kD1 : (pass == 1 ? kD2 : kD3)), tmem_base + kRHi,
                             tmem_base + kRLo, sbase + kTHi, sbase + kTLo, 0, kC * 128, 0, kC / 8,
                             tc::idesc_tf32(128, 64), pass, pass + 1);
            tc::mma_commit(&bars[2]);
        }
        __syncwarp();
        pend = 0x4u;
        const bool ok2 = tc::mbar_wait(&bars[2], ph, polls);   // agreed on before MMA-3 is issued
        tc::fence_after_sync();

        // ---- 3. Delta^T = sum of the three passes, split; Y_Q kept for the outputs ----
        float yq[32];
        tc::tmem_ld32(tm + kYQ + 32 * hf, yq);
#pragma unroll 1
        for (int grp = 0; grp < 4; ++grp) {
            float d1[8], d2[8], d3[8];
            tc::tmem_ld8(tm + kD1 + 32 * hf + 8 * grp, d1);
            tc::tmem_ld8(tm + kD2 + 32 * hf + 8 * grp, d2);
            tc::tmem_ld8(tm + kD3 + 32 * hf + 8 * grp, d3);
            tc::ld_wait();
            uint32_t hi[8], lo[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) tc::split_tf32(d1[e] + (d2[e] + d3[e]), hi[e], lo[e]);
            tc::tmem_st8(tm + kDtHi + 32 * hf + 8 * grp, hi);
            tc::tmem_st8(tm + kDtLo + 32 * hf + 8 * grp, lo);
        }
        tc::st_wait();

        // ---- MMA-3: [Z | (P Delta)^T] = Delta^T [Ktilde | P^T] (N = 192), two issuers ----
        tc::fence_before_sync();
        ok = __syncthreads_and(ok2) != 0;
        tc::fence_after_sync();
        if (!ok) break;
        if (tid == kIss0 || tid == kIss1) {       // over the first / second half of K (t)
            const bool first = tid == kIss0;
            mma_passes<true>(tmem_base + (first ? kM3a : kM3b), tmem_base + kDtHi, tmem_base + kDtLo, sbase + kBHi,
                             sbase + kBLo, 0, kBRows * 128, first ? 0 : kC / 16, first ? kC / 16 : kC / 8,
                             tc::idesc_tf32(128, kBRows), 0, 3);
            tc::mma_commit(&bars[3]);
        }
        __syncwarp();
        pend = 0x8u;
        // while MMA-3 runs: the next chunk's low parts of k-blocks 0-1 (columns 0-63), into T's space,
        // which MMA-2 no longer reads (k-blocks 2-3 lie under MMA-3's B operand and wait for the next
        // chunk's start); the chunk measured 2.418 -> 2.376 ms at batch 8, T 4096
        bool okl = true;
        lo_half = false;
        if (c0 + kC < T) {
            okl = tc::mbar_wait(&bars[4], kq_ph, copy_polls);
            if (okl) {
#pragma unroll 2
                for (int i = 0; i < 8; ++i) {
                    const uint32_t off = tc::sw128_offset(16 * warp + 2 * i + (lane >> 4), 4 * (lane & 15), 128);
                    const uint4 x = ld_shared_v4(sbase + kKQHi + off);
                    st_shared_v4(sbase + kKQLo + off, tf32_low(x.x), tf32_low(x.y), tf32_low(x.z), tf32_low(x.w));
                }
                lo_half = true;
            }
        }
        const bool ok3 = tc::mbar_wait(&bars[3], ph, polls);   // agreed on at the end of the chunk
        tc::fence_after_sync();

        // ---- 4. outputs and the new state ----
#pragma unroll
        for (int grp = 0; grp < 4; ++grp) {
            float pa[8], pb[8];
            tc::tmem_ld8(tm + kM3a + 128 + 32 * hf + 8 * grp, pa);
            tc::tmem_ld8(tm + kM3b + 128 + 32 * hf + 8 * grp, pb);
            tc::ld_wait();
            const int t0 = 32 * hf + 8 * grp;
            const float4 g_lo = *reinterpret_cast<const float4 *>(sc.gamma + t0);
            const float4 g_hi = *reinterpret_cast<const float4 *>(sc.gamma + t0 + 4);
            const float gm[8] = {g_lo.x, g_lo.y, g_lo.z, g_lo.w, g_hi.x, g_hi.y, g_hi.z, g_hi.w};
            if constexpr (TMA_O) {                      // o[t][a] into the tile, a = r: 128 B per warp store
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    st_shared_b32(sbase + kOStage + ((t0 + e) * kD + r) * 4,
                                  __float_as_uint(fmaf(gm[e], yq[8 * grp + e], pa[e] + pb[e]) * p.inv_sqrt_d));
            } else {
                float *op = obase + (int64_t)(c0 + t0) * p.o_stride + r;
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    if (t0 + e < n)
                        __stcs(op + (int64_t)e * p.o_stride,
                               fmaf(gm[e], yq[8 * grp + e], pa[e] + pb[e]) * p.inv_sqrt_d);
            }
        }
        if constexpr (TMA_O) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        {
            const float gC = sc.gamma[kC - 1];
#pragma unroll
            for (int cb = 0; cb < 2; ++cb) {
                float za[32], zb[32];
                tc::tmem_ld32(tm + kM3a + 64 * hf + 32 * cb, za);
                tc::tmem_ld32(tm + kM3b + 64 * hf + 32 * cb, zb);
                tc::ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j) S[32 * cb + j] = fmaf(gC, S[32 * cb + j], za[j] + zb[j]);
            }
        }
        tc::fence_before_sync();
        ok = __syncthreads_and(ok3 && okl) != 0;           // also: scalars and the operand buffer are reused
        tc::fence_after_sync();
        if (!ok) break;
        if (TMA_O && tid == 0) store_o_tile(&o_map, sbase + kOStage, h * kD, c0, seq);
        pend = 0;
        ph ^= 1u;
    }
    cp_async_wait<0>();                                    // no copy left in flight
    if (TMA_O && tid == 0) o_tile_done();
    if (!ok) {
        // a wait gave up: let the MMAs and tensor copies still in flight finish (again bounded) before
        // the memory they write is freed; count the event; the state of this head becomes NaN
#pragma unroll 1
        for (int i = 0; i < 4; ++i)
            if (pend & (1u << i)) tc::mbar_wait(&bars[i], ph, kWaitLimit);
        if (kq_pend) tc::mbar_wait(&bars[4], kq_ph, kWaitLimit);
        if (tid == 0) atomicAdd(&g_tc_wait_timeouts, 1u);
#pragma unroll
        for (int j = 0; j < 64; ++j) S[j] = __int_as_float(0x7fc00000);
    }
#pragma unroll
    for (int j = 0; j < 64; ++j) srow[j] = from_f32<TS>(S[j]);
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem_base, 512);
    }
}

std::atomic<uint32_t> g_wait_polls{kWaitLimit};        // the MMA waits' bound
std::atomic<uint32_t> g_copy_wait_polls{kWaitLimit};   // the tensor-copy waits' bound

// cuTensorMapEncodeTiled from the driver (through the runtime's entry-point query, so the library
// needs no link to the driver library); null if unavailable.
PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess || q != cudaDriverEntryPointSuccess)
            f = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }();
    return fn;
}

// The 3-D map of o for the tile store: (column < NV D, token < T, sequence < batch), box 128 x 64 x 1.
// False when o's layout does not allow it (base or row pitch not a multiple of 16 bytes) or the encoder
// is unavailable; the plain-store kernel then runs.
bool o_tensor_map(const PrefillParams &p, CUtensorMap *map)
{
    if (((uintptr_t)p.o & 15) != 0 || (p.o_stride & 3) != 0) return false;
    const PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (enc == nullptr) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)p.nv * kD, (cuuint64_t)p.seq_len, (cuuint64_t)p.batch};
    const cuuint64_t strides[2] = {(cuuint64_t)p.o_stride * 4, (cuuint64_t)p.o_stride * 4 * (cuuint64_t)p.seq_len};
    const cuuint32_t box[3] = {(cuuint32_t)kD, (cuuint32_t)kC, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, p.o, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

// The 3-D map of k or q for the chunk copies: (column < NK D, token < T, sequence < batch), box 32 x 64
// x 1 (128 bytes x 64 tokens) with the 128-byte swizzle; tokens past T read as zeros.  The caller
// guarantees a 16-byte aligned base and row pitch.
bool kq_tensor_map(const PrefillParams &p, const float *base, CUtensorMap *map)
{
    const PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (enc == nullptr) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)p.nk * kD, (cuuint64_t)p.seq_len, (cuuint64_t)p.batch};
    const cuuint64_t strides[2] = {(cuuint64_t)p.qk_stride * 4, (cuuint64_t)p.qk_stride * 4 * (cuuint64_t)p.seq_len};
    const cuuint32_t box[3] = {32, (cuuint32_t)kC, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename TS, bool TMA_O>
cudaError_t launch_kernel(const PrefillParams &p, const CUtensorMap &omap, const CUtensorMap &kmap,
                          const CUtensorMap &qmap, cudaStream_t s)
{
    constexpr auto kern = prefill_tc_d128<TS, TMA_O>;
    const cudaError_t e = allow_dynamic_smem<kern>((int)kSmemBytes);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)((int64_t)p.batch * p.nv), kThreads, kSmemBytes, s>>>(p, g_wait_polls.load(), g_copy_wait_polls.load(), omap,
                                                                          kmap, qmap);
    return cudaGetLastError();
}

template <typename TS>
cudaError_t launch_typed(const PrefillParams &p, cudaStream_t s)
{
    CUtensorMap kmap{}, qmap{}, omap{};
    if (!kq_tensor_map(p, p.k, &kmap) || !kq_tensor_map(p, p.q, &qmap)) return cudaErrorNotSupported;
    if (o_tensor_map(p, &omap)) return launch_kernel<TS, true>(p, omap, kmap, qmap, s);
    return launch_kernel<TS, false>(p, omap, kmap, qmap, s);
}

}  // namespace

cudaError_t launch_prefill_tc(const PrefillParams &p, bool f16_state, cudaStream_t s)
{
    return f16_state ? launch_typed<__half>(p, s) : launch_typed<float>(p, s);
}

void tc_set_wait_polls(uint32_t polls)
{
    g_wait_polls.store(polls);
    g_copy_wait_polls.store(polls);
}

void tc_set_mma_wait_polls(uint32_t polls) { g_wait_polls.store(polls); }

cudaError_t tc_wait_timeouts(unsigned *count)
{
    const cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return e;
    return cudaMemcpyFromSymbol(count, g_tc_wait_timeouts, sizeof(unsigned));
}

}  // namespace gdn
