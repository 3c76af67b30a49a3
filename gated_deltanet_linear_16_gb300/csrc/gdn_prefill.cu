// gdn_prefill.cu -- token-sequential prefill: seq_len tokens per sequence
// through the gated delta rule in one launch, the state held on chip.
//
// Follows metrale_model_layers/layers/ops/ssm_gdn_a.rs, launcher
// `gdn_prefill_regresident` (the recurrence walks the tokens in order, the
// state stays in registers, raw o for every token, no norm); the step itself
// is logicaffeine_compile/codegen_cuda/gdn.rs, kernel `gdn_step`.
//
// Rows of S never interact: row a needs only k, q, alpha, beta of the token
// and its own v[a].  So the GB300 kernel keeps the state in registers, 128
// fp32 per thread, for all tokens: each thread holds two rows x half of the
// columns, so
//  * every broadcast 16-byte shared-memory read of k or q feeds both rows
//    (half the shared loads of one-row-per-thread), and u = S[a].k,
//    o[a] = S_new[a].q need one shuffle each to add the two halves;
//  * o is read out of the updated state, o = S_new q / sqrt(D), which equals
//    (alpha w + coef kq)/sqrt(D) and needs no per-token k.q;
//  * the decay is deferred: the row is held as S = gam * R with a per-row
//    scalar gam (the product of the alphas since the last fold), so a token
//    costs three multiply-adds per element (u, the rank-1 write into R, o)
//    instead of four; gam is folded back into R before it could underflow
//    (below 2^-32, or alpha = 0).  The write into R needs coef / gam: it is
//    taken as coef * (1/gam), with 1/alpha computed once per staged token and
//    1/gam re-derived exactly at every chunk, so no division sits in the
//    token loop and the running reciprocal drifts over at most 8 tokens;
//  * the multiply-adds work on element pairs (float2) held in registers;
//  * a CTA is one warp (32 rows of one head).  With ~168 registers a thread
//    an SM holds 11-12 such warps, and one-warp CTAs let the block scheduler
//    spread the B*NV*D/32 warps evenly over the SMs (a 4-warp CTA per head
//    would leave some SMs with 3 heads and others with 2);
//  * an fp16 state is widened once when loaded and rounded to fp16 (nearest
//    even) once when stored: across the tokens it is carried in fp32;
//  * per-token inputs stream through a two-stage cp.async ring in shared
//    memory (8 tokens per stage), so the next chunk's loads overlap this
//    chunk's arithmetic.  cp.async waits are hardware group waits (no spin
//    loop on a flag).
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kD = 128;
constexpr int kTC = 8;            // tokens per stage
constexpr int kRows = 32;         // rows per CTA (one warp)

struct __align__(16) Stage {
    float k[kTC][kD];
    float q[kTC][kD];
    float v[kTC][kRows];
    float alpha[kTC];
    float beta[kTC];
    float inv_alpha[kTC];         // 1 / alpha, computed once per chunk after it lands
};

__device__ __forceinline__ void cp_async4(void *smem, const void *gmem) {
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(s), "l"(gmem) : "memory");
}

__device__ __forceinline__ float4 lds128(unsigned addr) {
    float4 r;
    asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];\n"
                 : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w) : "r"(addr));
    return r;
}

// `addr` made data-dependent on `dep` through a mask that is zero at run time
// but unknown to the compiler.  Without it the scheduler lifts the second
// pass's 64 shared loads above the first pass's reduction (they do not depend
// on coef) and the 128-register state row spills.
__device__ __forceinline__ unsigned after(unsigned addr, float dep, unsigned zero) {
    return addr + (__float_as_uint(dep) & zero);
}

// Stage tokens [t0, t0 + n) of this warp's (sequence, head, row block).  The
// loops stay rolled: they run while the 128 state registers are live, so they
// must not need many registers of their own.
__device__ __forceinline__ void stage_chunk(Stage &st, const PrefillParams &p, int seq, int h, int g,
                                            int r0, int t0, int n, int lane)
{
    const int64_t tok0 = (int64_t)seq * p.seq_len + t0;
    const float *kp = p.k + tok0 * p.qk_stride + (int64_t)g * kD + 4 * lane;
    const float *qp = p.q + tok0 * p.qk_stride + (int64_t)g * kD + 4 * lane;
#pragma unroll 1
    for (int tt = 0; tt < n; ++tt) {
        cp_async16(&st.k[tt][4 * lane], kp);
        cp_async16(&st.q[tt][4 * lane], qp);
        kp += p.qk_stride;
        qp += p.qk_stride;
    }
    // v: n tokens x 32 rows = n x 8 vectors of 16 bytes
#pragma unroll 1
    for (int c = lane; c < n * (kRows / 4); c += 32) {
        const int tt = c / (kRows / 4), part = c % (kRows / 4);
        cp_async16(&st.v[tt][4 * part], p.v + (tok0 + tt) * p.v_stride + (int64_t)h * kD + r0 + 4 * part);
    }
    if (lane < n) {
        cp_async4(&st.alpha[lane], p.alpha + (tok0 + lane) * p.gb_stride + h);
        cp_async4(&st.beta[lane], p.beta + (tok0 + lane) * p.gb_stride + h);
    }
}

// Element pairs through scalar fp32 FMA / multiply.  (The paired form,
// fma.rn.f32x2, gives the same bits; at this kernel's occupancy -- about ten
// warps per SM -- scalar FMA issues faster on GB300: 95 vs ~80 FMA per clock
// per SM in a pure FMA loop, 4.43 vs 4.50 ms here.)
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    return make_float2(__fmaf_rn(a.x, b.x, c.x), __fmaf_rn(a.y, b.y, c.y));
}
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
    return make_float2(__fmul_rn(a.x, b.x), __fmul_rn(a.y, b.y));
}

// Four consecutive state elements <-> fp32 (fp16: one 8-byte access, rounded to
// nearest even on the store).
__device__ __forceinline__ float4 load4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ float4 load4(const __half *p) {
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    const float2 a = Vec16<__half>::h2f(u.x), b = Vec16<__half>::h2f(u.y);
    return make_float4(a.x, a.y, b.x, b.y);
}
__device__ __forceinline__ void store4(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }
__device__ __forceinline__ void store4(__half *p, float4 v) {
    *reinterpret_cast<uint2 *>(p) = make_uint2(Vec16<__half>::f2h(v.x, v.y), Vec16<__half>::f2h(v.z, v.w));
}

// Smallest scale kept deferred before it is folded back into the stored row.
constexpr float kMinScale = 0x1p-32f;

template <typename TS>
__global__ void __launch_bounds__(kRows, 12)
prefill_d128(const PrefillParams p)
{
    __shared__ Stage ring[2];

    const int lane = threadIdx.x;
    const int half = lane >> 4;                        // which half of the columns
    const int pr = lane & 15;                          // which pair of rows
    const int blocks_per_head = kD / kRows;            // 4
    const int head = blockIdx.x / blocks_per_head;     // (sequence, value head)
    const int r0 = (blockIdx.x - head * blocks_per_head) * kRows;
    const int seq = head / p.nv;
    const int h = head - seq * p.nv;
    const int g = h % p.nk;
    const int a0 = r0 + 2 * pr;                        // this thread's rows: a0, a0 + 1

    const int T = p.seq_len;
    const int nchunks = (T + kTC - 1) / kTC;
    stage_chunk(ring[0], p, seq, h, g, r0, 0, min(kTC, T), lane);   // before the state is live
    cp_async_commit();

    // Two rows x 64 columns per thread: columns 4c..4c+3 for c = 2 jj + half, jj = 0..15, so a
    // warp-wide 16-byte shared load serves both rows of a thread and touches two distinct
    // 16-byte chunks in different banks.  Rows are held as S = gam * R (deferred decay).
    TS *row = reinterpret_cast<TS *>(p.state) + seq * p.pitch + (int64_t)h * kD * kD + (int64_t)a0 * kD;
    float2 R[2][kD / 4];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
#pragma unroll
        for (int jj = 0; jj < kD / 8; ++jj) {
            const float4 t = load4(row + rr * kD + 4 * (2 * jj + half));
            R[rr][2 * jj] = make_float2(t.x, t.y);
            R[rr][2 * jj + 1] = make_float2(t.z, t.w);
        }
    }
    float gam = 1.0f, inv_gam = 1.0f;

    float *orow = p.o + (int64_t)seq * T * p.o_stride + (int64_t)h * kD + a0 + half;
    const unsigned lane_off = 16u * half;
    for (int c = 0; c < nchunks; ++c) {
        if (c + 1 < nchunks) {
            const int t1 = (c + 1) * kTC;
            stage_chunk(ring[(c + 1) & 1], p, seq, h, g, r0, t1, min(kTC, T - t1), lane);
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncwarp();
        Stage &st = ring[c & 1];
        const int n = min(kTC, T - c * kTC);
        if (lane < n) st.inv_alpha[lane] = 1.0f / st.alpha[lane];
        inv_gam = 1.0f / gam;          // exact once a chunk: the running product drifts at most 8 steps
        __syncwarp();
        const unsigned k_s = (unsigned)__cvta_generic_to_shared(st.k[0]) + lane_off;
        const unsigned q_s = (unsigned)__cvta_generic_to_shared(st.q[0]) + lane_off;
        for (int tt = 0; tt < n; ++tt) {
            const unsigned kt = k_s + tt * (kD * 4), qt = q_s + tt * (kD * 4);
            float2 ua0 = make_float2(0.f, 0.f), ua1 = ua0, ub0 = ua0, ub1 = ua0;
#pragma unroll
            for (int jj = 0; jj < kD / 8; ++jj) {
                const float4 kk = lds128(kt + 32 * jj);
                const float2 k01 = make_float2(kk.x, kk.y), k23 = make_float2(kk.z, kk.w);
                ua0 = ffma2(R[0][2 * jj], k01, ua0);
                ua1 = ffma2(R[0][2 * jj + 1], k23, ua1);
                ub0 = ffma2(R[1][2 * jj], k01, ub0);
                ub1 = ffma2(R[1][2 * jj + 1], k23, ub1);
            }
            float pa = (ua0.x + ua0.y) + (ua1.x + ua1.y);
            float pb = (ub0.x + ub0.y) + (ub1.x + ub1.y);
            pa += __shfl_xor_sync(kFull, pa, 16);
            pb += __shfl_xor_sync(kFull, pb, 16);
            const float alpha = st.alpha[tt], beta = st.beta[tt];
            const float coef_a = beta * (st.v[tt][2 * pr] - alpha * (gam * pa));
            const float coef_b = beta * (st.v[tt][2 * pr + 1] - alpha * (gam * pb));
            const float gnew = alpha * gam;
            const unsigned k2 = after(kt, coef_a, p.zero), q2 = after(qt, coef_b, p.zero);
            float2 oa0 = make_float2(0.f, 0.f), oa1 = oa0, ob0 = oa0, ob1 = oa0;
            if (gnew >= kMinScale) {            // warp-uniform: one head per warp
                const float inv_gnew = inv_gam * st.inv_alpha[tt];
                const float ca = coef_a * inv_gnew, cb = coef_b * inv_gnew;
                const float2 ca2 = make_float2(ca, ca), cb2 = make_float2(cb, cb);
#pragma unroll
                for (int jj = 0; jj < kD / 8; ++jj) {
                    const float4 kk = lds128(k2 + 32 * jj), qq = lds128(q2 + 32 * jj);
                    const float2 k01 = make_float2(kk.x, kk.y), k23 = make_float2(kk.z, kk.w);
                    const float2 q01 = make_float2(qq.x, qq.y), q23 = make_float2(qq.z, qq.w);
                    R[0][2 * jj] = ffma2(ca2, k01, R[0][2 * jj]);
                    R[0][2 * jj + 1] = ffma2(ca2, k23, R[0][2 * jj + 1]);
                    R[1][2 * jj] = ffma2(cb2, k01, R[1][2 * jj]);
                    R[1][2 * jj + 1] = ffma2(cb2, k23, R[1][2 * jj + 1]);
                    oa0 = ffma2(R[0][2 * jj], q01, oa0);
                    oa1 = ffma2(R[0][2 * jj + 1], q23, oa1);
                    ob0 = ffma2(R[1][2 * jj], q01, ob0);
                    ob1 = ffma2(R[1][2 * jj + 1], q23, ob1);
                }
                gam = gnew;
                inv_gam = inv_gnew;
            } else {
                const float2 g2 = make_float2(gnew, gnew);
                const float2 ca2 = make_float2(coef_a, coef_a), cb2 = make_float2(coef_b, coef_b);
#pragma unroll
                for (int jj = 0; jj < kD / 8; ++jj) {
                    const float4 kk = lds128(k2 + 32 * jj), qq = lds128(q2 + 32 * jj);
                    const float2 k01 = make_float2(kk.x, kk.y), k23 = make_float2(kk.z, kk.w);
                    const float2 q01 = make_float2(qq.x, qq.y), q23 = make_float2(qq.z, qq.w);
                    R[0][2 * jj] = ffma2(ca2, k01, fmul2(g2, R[0][2 * jj]));
                    R[0][2 * jj + 1] = ffma2(ca2, k23, fmul2(g2, R[0][2 * jj + 1]));
                    R[1][2 * jj] = ffma2(cb2, k01, fmul2(g2, R[1][2 * jj]));
                    R[1][2 * jj + 1] = ffma2(cb2, k23, fmul2(g2, R[1][2 * jj + 1]));
                    oa0 = ffma2(R[0][2 * jj], q01, oa0);
                    oa1 = ffma2(R[0][2 * jj + 1], q23, oa1);
                    ob0 = ffma2(R[1][2 * jj], q01, ob0);
                    ob1 = ffma2(R[1][2 * jj + 1], q23, ob1);
                }
                gam = 1.0f;
                inv_gam = 1.0f;
            }
            float sa = (oa0.x + oa0.y) + (oa1.x + oa1.y);
            float sb = (ob0.x + ob0.y) + (ob1.x + ob1.y);
            sa += __shfl_xor_sync(kFull, sa, 16);
            sb += __shfl_xor_sync(kFull, sb, 16);
            const float o = gam * (half ? sb : sa);     // lane pr stores row a0, lane 16 + pr row a0 + 1
            __stcs(orow + (int64_t)(c * kTC + tt) * p.o_stride, o * p.inv_sqrt_d);
        }
        __syncwarp();
    }

#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
#pragma unroll
        for (int jj = 0; jj < kD / 8; ++jj)
            store4(row + rr * kD + 4 * (2 * jj + half),
                   make_float4(gam * R[rr][2 * jj].x, gam * R[rr][2 * jj].y,
                               gam * R[rr][2 * jj + 1].x, gam * R[rr][2 * jj + 1].y));
    }
}

// Any D <= 256 and any alignment: one CTA per (sequence, head), one warp per
// row (rows strided over 4 warps), lanes strided over columns with the row in
// registers for all tokens; token inputs read straight from global memory.
constexpr int kGenWarps = 4;
constexpr int kMaxD = 256;

template <typename TS>
__global__ void __launch_bounds__(kGenWarps * 32)
prefill_generic(const PrefillParams p)
{
    constexpr int MAXV = kMaxD / 32;
    const int D = p.d;
    const int seq = blockIdx.x / p.nv;
    const int h = blockIdx.x - seq * p.nv;
    const int g = h % p.nk;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int T = p.seq_len;

    for (int a = warp; a < D; a += kGenWarps) {
        TS *row = reinterpret_cast<TS *>(p.state) + seq * p.pitch + (int64_t)h * D * D + (int64_t)a * D;
        float s[MAXV];
#pragma unroll
        for (int j = 0; j < MAXV; ++j) {
            const int c = lane + 32 * j;
            s[j] = c < D ? to_f32<TS>(row[c]) : 0.f;
        }
        for (int t = 0; t < T; ++t) {
            const int64_t tok = (int64_t)seq * T + t;
            const float *kp = p.k + tok * p.qk_stride + (int64_t)g * D;
            const float *qp = p.q + tok * p.qk_stride + (int64_t)g * D;
            float kr[MAXV];
            float u = 0.f;
#pragma unroll
            for (int j = 0; j < MAXV; ++j) {
                const int c = lane + 32 * j;
                kr[j] = c < D ? kp[c] : 0.f;
                u = fmaf(s[j], kr[j], u);
            }
            u = group_sum<32>(u);
            const float alpha = p.alpha[tok * p.gb_stride + h];
            const float beta = p.beta[tok * p.gb_stride + h];
            const float coef = beta * (p.v[tok * p.v_stride + (int64_t)h * D + a] - alpha * u);
            float w = 0.f;
#pragma unroll
            for (int j = 0; j < MAXV; ++j) {
                const int c = lane + 32 * j;
                s[j] = fmaf(coef, kr[j], alpha * s[j]);
                if (c < D) w = fmaf(s[j], qp[c], w);
            }
            w = group_sum<32>(w);
            if (lane == 0) p.o[tok * p.o_stride + (int64_t)h * D + a] = w * p.inv_sqrt_d;
        }
#pragma unroll
        for (int j = 0; j < MAXV; ++j) {
            const int c = lane + 32 * j;
            if (c < D) row[c] = from_f32<TS>(s[j]);
        }
    }
}

template <typename TS>
cudaError_t launch_typed(const PrefillParams &p, bool fast, cudaStream_t s)
{
    const int64_t heads = (int64_t)p.batch * p.nv;
    if (fast) {
        prefill_d128<TS><<<(unsigned)(heads * (kD / kRows)), kRows, 0, s>>>(p);
    } else {
        prefill_generic<TS><<<(unsigned)heads, kGenWarps * 32, 0, s>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const PrefillParams &p, bool f16_state, bool fast, cudaStream_t s)
{
    return f16_state ? launch_typed<__half>(p, fast, s) : launch_typed<float>(p, fast, s);
}

}  // namespace gdn
