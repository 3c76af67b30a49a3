// gdn_norm.cu -- the gated RMS norm as its own launch, over rows of raw
// outputs o (e.g. every token of a prefill call), with a bf16 output or the
// int8 activation groups.
//
// Follows logicaffeine_compile/codegen_cuda/gdn.rs, kernels `gdn_gate_norm`
// (out = gn o / sqrt(mean_head o^2 + eps) * silu(z): the norm first, then the
// gate; gn shared by all heads) and `gdn_gate_norm_q` (the same with the
// int8 quantisation of the o-projection's input fused in: groups of 32 values,
// scale = max |y| / 127, codes rounded to nearest even).
//
// An HBM stream (o and z read once, the output written once).  General D: one
// warp per (row, head), lanes strided over the head's D values (coalesced
// 128-byte warp accesses), every load of a lane in flight before the
// reduction; 8 warps per CTA.  D == 128 with aligned rows takes the vector
// kernels below: gate_norm_d128 (bf16) and gate_norm_q8_hw (int8).
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kWarpsPerCta = 8;
constexpr int kMaxPer = 8;                 // D <= 256: values per lane

// y / s rounded to nearest (the IEEE quotient) from r = 1/s (the IEEE
// reciprocal), by Markstein's correction (P. Markstein, "Computation of
// elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
// Dev. 34(1), 1990): q0 = RN(y r), e = y - s q0 (exact in one FMA), q =
// RN(q0 + e r).  The theorem gives RN(y / s) when r is within half an ulp of
// 1/s and q0 within an ulp of y/s, with no underflow; the residual e is about
// |y/s| 2^-24 s, so it stays normal for s >= 2^-60 whenever the quotient is
// large enough to matter for an int8 code (a smaller one rounds to 0 either
// way).  Checked on a GB300 against the IEEE division bit for bit: every float
// y in [s/4, 127.5 s] for 256 random scales (19.3e9 quotients, no difference)
// and 2.55e9 random pairs over scales from 2^-107 (two quotients differed,
// both with s near 1e-32 and codes 0; those scales take the division).
constexpr float kMinCorrectedScale = 0x1p-60f;
// Adding 1.5 x 2^23 to a float q with |q| < 2^22 rounds it to an integer n, to nearest with ties to
// even as __float2int_rn does, and leaves n in the low bits of the sum's encoding (0x4B400000 + n), so
// the sum's low byte is n's two's-complement byte: the int8 code, by one add instead of a conversion
// (whose lower throughput measured ~1 % of this kernel's time; the same codes).
constexpr float kRoundToInt = 12582912.0f;
__device__ __forceinline__ float quotient_rn(float y, float s, float r)
{
    const float q0 = __fmul_rn(y, r);
    return __fmaf_rn(__fmaf_rn(-q0, s, y), r, q0);
}

// silu with the fast division (within 2 ulp): this kernel is an elementwise
// stream, where the IEEE division of the gate cost 7 % of the time.  An int8
// code is still that of the IEEE quotient (quotient_rn).
__device__ __forceinline__ float silu_fast(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

template <int EPI>
__global__ void __launch_bounds__(kWarpsPerCta * 32)
gate_norm_rows(const NormParams p)
{
    const int lane = threadIdx.x & 31;
    const int64_t unit = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);   // (row, head)
    if (unit >= p.rows * p.nv) return;                  // whole warps leave together
    const int64_t row = unit / p.nv;
    const int h = (int)(unit - row * p.nv);
    const int D = p.d;
    const float *op = p.o + row * p.o_stride + (int64_t)h * D;
    const float *zp = p.z + row * p.z_stride + (int64_t)h * D;

    float ov[kMaxPer], zv[kMaxPer];
#pragma unroll
    for (int j = 0; j < kMaxPer; ++j) {
        const int a = lane + 32 * j;
        ov[j] = a < D ? __ldcs(op + a) : 0.f;
        zv[j] = a < D ? __ldcs(zp + a) : 0.f;
    }
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxPer; ++j) ss = fmaf(ov[j], ov[j], ss);
    ss = group_sum<32>(ss);
    const float rstd = rsqrtf(ss / (float)D + p.eps);

#pragma unroll
    for (int j = 0; j < kMaxPer; ++j) {
        if (32 * j >= D) break;                         // warp-uniform
        const int a = lane + 32 * j;
        const bool in = a < D;
        const float y = in ? __ldg(p.gn + a) * ov[j] * rstd * silu_fast(zv[j]) : 0.f;
        if constexpr (EPI == kEpiBf16) {
            if (in) p.out[row * p.out_stride + (int64_t)h * D + a] = bf16_bits_rn(y);
        } else {                                        // D % 32 == 0: a whole group per j
            if (p.y != nullptr) p.y[row * p.y_stride + (int64_t)h * D + a] = y;
            quant_group32(y, p.xq + row * p.xq_stride + (int64_t)h * D + a,
                          p.xs + row * p.xs_stride + (int64_t)h * (D / 32) + j, lane);
        }
    }
}

// D == 128 with 16-byte aligned rows, bf16 output: a lane holds 4 consecutive
// values of a head (one 16-byte load each of o and z), warps loop over (row,
// head) units with several units in flight, and the grid is a few CTAs per SM.
// (The int8 output takes gate_norm_q8_hw below.)
constexpr int kD = 128;
constexpr int kCtasPerSm = 8;
// (row, head) units a warp has in flight: 4 (measured 312 us against 324 with 2
// and 371 with 1 over 32768 rows x 48 heads).
template <int EPI> constexpr int kInFlight = 4;   // (bf16 only)

template <int EPI>
__device__ __forceinline__ void norm_unit_d128(const NormParams &p, int64_t row, int h, float4 ov, float4 zv,
                                               int lane)
{
    static_assert(EPI == kEpiBf16, "the vector kernel's int8 output is gate_norm_q8_hw");
    float ss = ov.x * ov.x;
    ss = fmaf(ov.y, ov.y, ss);
    ss = fmaf(ov.z, ov.z, ss);
    ss = fmaf(ov.w, ov.w, ss);
    ss = group_sum<32>(ss);
    const float rstd = rsqrtf(ss * (1.0f / kD) + p.eps);
    const float4 g = __ldg(reinterpret_cast<const float4 *>(p.gn) + lane);
    float y[4] = {g.x * ov.x * rstd * silu_fast(zv.x), g.y * ov.y * rstd * silu_fast(zv.y),
                  g.z * ov.z * rstd * silu_fast(zv.z), g.w * ov.w * rstd * silu_fast(zv.w)};
    const int64_t e0 = (int64_t)h * kD + 4 * lane;
    const uint2 b = make_uint2((unsigned)bf16_bits_rn(y[0]) | ((unsigned)bf16_bits_rn(y[1]) << 16),
                               (unsigned)bf16_bits_rn(y[2]) | ((unsigned)bf16_bits_rn(y[3]) << 16));
    __stcs(reinterpret_cast<uint2 *>(p.out + row * p.out_stride + e0), b);
}

// Each warp takes chunks of NF consecutive (row, head) units, chunks nwarps
// apart.  Positions advance by a precomputed (rows, heads) stride and by one
// head within a chunk, so the only 64-bit division is the first one (a
// division per unit had made the int8 kernel 10 % slower).
template <int EPI>
__global__ void __launch_bounds__(kWarpsPerCta * 32)
gate_norm_d128(const NormParams p)
{
    constexpr int NF = kInFlight<EPI>;
    const int lane = threadIdx.x & 31;
    const int64_t units = p.rows * p.nv;
    const int64_t stride = (int64_t)gridDim.x * kWarpsPerCta * NF;    // units between a warp's chunks
    int64_t u = ((int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5)) * NF;
    if (u >= units) return;                             // whole warps leave together
    const int64_t step_rows = stride / p.nv;
    const int step_h = (int)(stride - step_rows * p.nv);
    int64_t row = u / p.nv;
    int h = (int)(u - row * p.nv);
    for (; u < units; u += stride) {
        float4 ov[NF], zv[NF];
        int64_t r = row;
        int hh = h;
#pragma unroll
        for (int i = 0; i < NF; ++i) {                  // every load of the chunk in flight
            ov[i] = zv[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (u + i < units) {
                const int64_t e0 = (int64_t)hh * kD + 4 * lane;
                ov[i] = __ldcs(reinterpret_cast<const float4 *>(p.o + r * p.o_stride + e0));
                zv[i] = __ldcs(reinterpret_cast<const float4 *>(p.z + r * p.z_stride + e0));
            }
            if (++hh == p.nv) { hh = 0; ++r; }
        }
        r = row;
        hh = h;
#pragma unroll
        for (int i = 0; i < NF; ++i) {
            if (u + i < units) norm_unit_d128<EPI>(p, r, hh, ov[i], zv[i], lane);
            if (++hh == p.nv) { hh = 0; ++r; }
        }
        row += step_rows;
        h += step_h;
        if (h >= p.nv) { h -= p.nv; ++row; }
    }
}

// int8 output: a quarter-warp (8 lanes) per (row, head) unit, 16 consecutive
// values a lane (four 16-byte loads each of o and z), so a warp works on four
// units at once and an int8 group of 32 values is 2 lanes.  A warp takes runs
// of 4 consecutive units, runs a grid apart.  Against the bf16 kernel's layout
// (a warp per unit, 4 values a lane) this cuts the per-unit reductions, the
// address and loop work per value: 304 us over 32768 rows x 48 heads, against
// 315 with a half-warp per unit and 365 with a warp.  A code is y / scale
// rounded, the IEEE quotient as the page decides codes, here by the corrected
// reciprocal (quotient_rn) instead of 16 divisions a lane.
__global__ void __launch_bounds__(kWarpsPerCta * 32)
gate_norm_q8_hw(const NormParams p)
{
    const int lane = threadIdx.x & 31;
    const int qw = lane >> 3, l = lane & 7;
    const int64_t units = p.rows * p.nv;
    const int64_t stride = (int64_t)gridDim.x * kWarpsPerCta * 4;
    int64_t u = ((int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5)) * 4;
    if (u >= units) return;
    const int64_t step_rows = stride / p.nv;
    const int step_h = (int)(stride - step_rows * p.nv);
    int64_t row = u / p.nv;
    int h = (int)(u - row * p.nv);
    float gv[16];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float4 g = __ldg(reinterpret_cast<const float4 *>(p.gn) + 4 * l + k);
        gv[4 * k] = g.x; gv[4 * k + 1] = g.y; gv[4 * k + 2] = g.z; gv[4 * k + 3] = g.w;
    }
    for (; u < units; u += stride) {
        int64_t r = row;
        int hh = h + qw;
        while (hh >= p.nv) { hh -= p.nv; ++r; }     // at most 3 steps (NV may be below 4)
        const bool active = u + qw < units;
        const int64_t e0 = (int64_t)hh * kD + 16 * l;
        float ov[16], zv[16];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
            if (active) {
                a = __ldcs(reinterpret_cast<const float4 *>(p.o + r * p.o_stride + e0) + k);
                b = __ldcs(reinterpret_cast<const float4 *>(p.z + r * p.z_stride + e0) + k);
            }
            ov[4 * k] = a.x; ov[4 * k + 1] = a.y; ov[4 * k + 2] = a.z; ov[4 * k + 3] = a.w;
            zv[4 * k] = b.x; zv[4 * k + 1] = b.y; zv[4 * k + 2] = b.z; zv[4 * k + 3] = b.w;
        }
        float ss = ov[0] * ov[0];
#pragma unroll
        for (int i = 1; i < 16; ++i) ss = fmaf(ov[i], ov[i], ss);
        ss = group_sum<8>(ss);
        const float rstd = rsqrtf(ss * (1.0f / kD) + p.eps);
        float y[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) y[i] = gv[i] * ov[i] * rstd * silu_fast(zv[i]);
        if (active && p.y != nullptr) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
                __stcs(reinterpret_cast<float4 *>(p.y + r * p.y_stride + e0) + k,
                       make_float4(y[4 * k], y[4 * k + 1], y[4 * k + 2], y[4 * k + 3]));
        }
        float am = fabsf(y[0]);
#pragma unroll
        for (int i = 1; i < 16; ++i) am = fmaxf(am, fabsf(y[i]));
        am = fmaxf(am, __shfl_xor_sync(kFull, am, 1));    // a group of 32 is 2 lanes
        const float sc = am > 0.f ? am / 127.0f : 1.0f;
        unsigned w[4] = {0u, 0u, 0u, 0u};
        if (sc >= kMinCorrectedScale) {                  // the quotients by Markstein's correction
            const float rs = 1.0f / sc;
#pragma unroll
            for (int i = 0; i < 16; ++i)   // the code byte: see kRoundToInt
                w[i >> 2] |= (__float_as_uint(__fadd_rn(quotient_rn(y[i], sc, rs), kRoundToInt)) & 0xffu) << (8 * (i & 3));
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) w[i >> 2] |= ((unsigned)(__float2int_rn(y[i] / sc) & 0xff)) << (8 * (i & 3));
        }
        if (active) {
            unsigned *q = reinterpret_cast<unsigned *>(p.xq + r * p.xq_stride + e0);
#pragma unroll
            for (int k = 0; k < 4; ++k) q[k] = w[k];
            if ((l & 1) == 0) p.xs[r * p.xs_stride + (int64_t)hh * (kD / 32) + (l >> 1)] = sc;
        }
        row += step_rows;
        h += step_h;
        if (h >= p.nv) { h -= p.nv; ++row; }
    }
}

}  // namespace

cudaError_t launch_gate_norm(const NormParams &p, int epi, bool fast, cudaStream_t s)
{
    const int64_t units = p.rows * p.nv;
    if (fast) {                                         // a warp takes 4 units at a time
        const int64_t full = (int64_t)sm_count() * kCtasPerSm;
        const int per_warp = epi == kEpiQ8 ? 4 : kInFlight<kEpiBf16>;
        const int64_t need = ((units + per_warp - 1) / per_warp + kWarpsPerCta - 1) / kWarpsPerCta;
        const unsigned grid = (unsigned)(need < full ? need : full);
        if (epi == kEpiQ8) gate_norm_q8_hw<<<grid, kWarpsPerCta * 32, 0, s>>>(p);
        else gate_norm_d128<kEpiBf16><<<grid, kWarpsPerCta * 32, 0, s>>>(p);
        return cudaGetLastError();
    }
    const unsigned grid = (unsigned)((units + kWarpsPerCta - 1) / kWarpsPerCta);
    if (epi == kEpiQ8) gate_norm_rows<kEpiQ8><<<grid, kWarpsPerCta * 32, 0, s>>>(p);
    else gate_norm_rows<kEpiBf16><<<grid, kWarpsPerCta * 32, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace gdn
