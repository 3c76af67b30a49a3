// gdn_decode.cu -- single-token gated delta rule kernels (raw fp32 output, or
// the gated RMS norm fused in the same CTA with a bf16 output), for fp32 and
// fp16 h-states.
//
// The step (logicaffeine_compile/codegen_cuda/gdn.rs, kernel `gdn_step`), for
// value head h, key/query head g = h mod NK and state row a:
//   u = S[a].k, w = S[a].q, kq = k.q, coef = beta (v[a] - alpha u),
//   o[a] = (alpha w + coef kq) / sqrt(D),  S[a][c] <- alpha S[a][c] + coef k[c].
// The norm (same page, kernel `gdn_gate_norm`): out = gn o / sqrt(mean o^2 + eps)
// * silu(z).  The fused variants follow metrale_model_layers/layers/ops/
// ssm_gdn_a.rs (`gdn_decode_f32_strided_norm`, `gdn_decode_f16_strided_norm`):
// the norm runs in the CTA that owns the head and only bf16 leaves the chip.
//
// GB300 design.  The state is ~99% of the bytes and is touched exactly once
// (one read, one write per element), so the kernel is an HBM stream:
//  * one CTA owns one (sequence, head) -- 8 warps x 16 rows -- so the norm's
//    reduction over the head's D outputs needs a single __syncthreads;
//  * every state access is a 16-byte vector: an fp32 row (512 B) is one
//    warp-wide load, an fp16 row (256 B) half of one, so a warp touches whole
//    128-byte lines and stores never leave partial sectors;
//  * each lane's state loads are issued in batches, the next batch in flight
//    while the current one is computed and written back, with 3-4 CTAs per
//    SM: some 50-100 KB of loads outstanding per SM, enough to cover HBM
//    latency at full bandwidth while the stores of earlier rows drain;
//  * k and q are read as this lane's own 16-byte columns, v/z/gn as one
//    coalesced read per warp (a float per row) that lanes broadcast by shuffle;
//  * the three dot products are butterfly shuffles inside the group of lanes
//    that holds a row (32 lanes fp32, 16 lanes fp16); k.q is reduced once per
//    warp, not per row.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kD = 128;

// ------------------------------------------------------------------ D == 128

// Shape of the D == 128 kernel: WARPS warps share one head (128 / WARPS rows
// each); each lane's state loads are issued in NB batches, batch b + 1 in
// flight while batch b is computed (NB == 1: everything in flight at once).
// Chosen by measurement on GB300 (48-layer fp32 workload, 256-slot fp16 pool):
// fp32 8 warps x 16 rows, 4 batches of 4 loads, 3 CTAs per SM; fp16 8 warps x
// 16 rows, 2 batches of 4 loads, 4 CTAs per SM.
// kSplit > 1 spreads a head over a cluster of kSplit CTAs (shorter CTAs, a
// shorter drain at the end of a launch); the fused norm then adds the CTAs'
// partial sums of squares over distributed shared memory in rank order.
template <typename TS> struct FastShape {
    static constexpr int kWarps = 8, kBatches = 4, kMinBlocks = 3, kSplit = 1;
};
template <> struct FastShape<__half> {
    static constexpr int kWarps = 8, kBatches = 2, kMinBlocks = 4, kSplit = 1;
};

template <typename TS, bool NORM, int WARPS, int NB, int MINB, int SPLIT>
__global__ void __launch_bounds__(WARPS * 32, MINB)
decode_d128(const DecodeParams p)
{
    using V = Vec16<TS>;
    constexpr int EPV = V::N;                  // state elements per 16-byte vector
    constexpr int LPR = kD / EPV;              // lanes per state row: 32 fp32, 16 fp16
    constexpr int RPL = 32 / LPR;              // rows per warp-wide load: 1 fp32, 2 fp16
    constexpr int RPW = kD / (WARPS * SPLIT);  // rows per warp
    constexpr int NLD = RPW / RPL;             // 16-byte state loads per lane
    constexpr int LPB = NLD / NB;              // loads per batch
    static_assert(RPW <= 32 && NLD % NB == 0 && NLD >= NB, "shape");

    const int unit = blockIdx.x / SPLIT;       // (sequence, value head)
    const int part = blockIdx.x - unit * SPLIT;  // which rows of the head (cluster rank)
    const int seq = unit / p.nv;
    const int h = unit - seq * p.nv;
    const int g = h % p.nk;                    // tiled key-head pairing
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int sub = lane / LPR;                // which row of a warp-wide load
    const int col = (lane % LPR) * EPV;        // first column this lane owns
    const int row0 = part * (kD / SPLIT) + warp * RPW;

    TS *S = reinterpret_cast<TS *>(p.state) + seq * p.pitch + (int64_t)h * kD * kD;
    TS *rowp = S + (int64_t)(row0 + sub) * kD + col;

    // 1. the first batch of this lane's state slice, in flight before anything else
    uint4 raw[NB > 1 ? 2 : 1][LPB];
#pragma unroll
    for (int i = 0; i < LPB; ++i) raw[0][i] = ld_stream16(rowp + (int64_t)i * RPL * kD);

    // 2. token inputs
    const float *kp = p.k + seq * p.qk_stride + (int64_t)g * kD + col;
    const float *qp = p.q + seq * p.qk_stride + (int64_t)g * kD + col;
    float kx[EPV], qx[EPV];
#pragma unroll
    for (int j = 0; j < EPV; j += 4) {
        const float4 a = ld_ro_f4(kp + j), b = ld_ro_f4(qp + j);
        kx[j] = a.x; kx[j + 1] = a.y; kx[j + 2] = a.z; kx[j + 3] = a.w;
        qx[j] = b.x; qx[j + 1] = b.y; qx[j + 2] = b.z; qx[j + 3] = b.w;
    }
    const bool row_lane = lane < RPW;          // lane r carries row row0 + r
    const float v_l = row_lane ? __ldg(p.v + seq * p.v_stride + (int64_t)h * kD + row0 + lane) : 0.f;
    float z_l = 0.f, gn_l = 0.f;
    if (NORM && row_lane) {
        z_l = __ldg(p.z + seq * p.z_stride + (int64_t)h * kD + row0 + lane);
        gn_l = __ldg(p.gn + row0 + lane);
    }
    const float alpha = __ldg(p.alpha + seq * p.gb_stride + h);
    const float beta = __ldg(p.beta + seq * p.gb_stride + h);

    float kq = 0.f;
#pragma unroll
    for (int j = 0; j < EPV; ++j) kq = fmaf(kx[j], qx[j], kq);
    kq = group_sum<LPR>(kq);

    // 3. per row: two dot products, the delta coefficient, output, write-back
    float o_keep = 0.f;                        // lane r keeps o of row row0 + r
#pragma unroll
    for (int bt = 0; bt < NB; ++bt) {
        if (bt + 1 < NB) {
#pragma unroll
            for (int i = 0; i < LPB; ++i)
                raw[(bt + 1) & 1][i] = ld_stream16(rowp + (int64_t)((bt + 1) * LPB + i) * RPL * kD);
        }
#pragma unroll
        for (int ii = 0; ii < LPB; ++ii) {
            const int i = bt * LPB + ii;       // load index within the lane's slice
            float s[EPV];
            V::unpack(raw[bt & 1][ii], s);
            float u = 0.f, w = 0.f;
#pragma unroll
            for (int j = 0; j < EPV; ++j) { u = fmaf(s[j], kx[j], u); w = fmaf(s[j], qx[j], w); }
            u = group_sum<LPR>(u);
            w = group_sum<LPR>(w);
            const float va = __shfl_sync(kFull, v_l, i * RPL + sub);
            const float coef = beta * (va - alpha * u);
            const float oa = (alpha * w + coef * kq) * p.inv_sqrt_d;
#pragma unroll
            for (int j = 0; j < EPV; ++j) s[j] = fmaf(coef, kx[j], alpha * s[j]);
            st_stream16(rowp + (int64_t)i * RPL * kD, V::pack(s));
            if constexpr (RPL == 1) {
                if (lane == i) o_keep = oa;
            } else {
#pragma unroll
                for (int r = 0; r < RPL; ++r) {
                    const float orr = __shfl_sync(kFull, oa, r * LPR);
                    if (lane == i * RPL + r) o_keep = orr;
                }
            }
        }
    }

    if constexpr (!NORM) {
        if (row_lane) p.o[seq * p.o_stride + (int64_t)h * kD + row0 + lane] = o_keep;
    } else {
        // 4. gated RMS norm over the head's 128 outputs, in this CTA (and its cluster peers)
        __shared__ float red[WARPS];
        __shared__ float part_sum;
        const float ss = group_sum<32>(o_keep * o_keep);   // lanes >= RPW hold 0
        if (lane == 0) red[warp] = ss;
        __syncthreads();
        float tot = 0.f;
#pragma unroll
        for (int i = 0; i < WARPS; ++i) tot += red[i];
        if constexpr (SPLIT > 1) {
            if (threadIdx.x == 0) part_sum = tot;
            cluster_arrive();
            cluster_wait();                    // every CTA's partial sum is written
            tot = 0.f;
#pragma unroll
            for (int r = 0; r < SPLIT; ++r) tot += ld_cluster_f32(&part_sum, r);
            cluster_arrive();                  // done reading the peers' shared memory
        }
        const float rstd = rsqrtf(tot * (1.0f / kD) + p.eps);
        if (row_lane) {
            const float y = gn_l * o_keep * rstd * silu(z_l);
            p.out[seq * p.out_stride + (int64_t)h * kD + row0 + lane] = bf16_bits_rn(y);
        }
        if constexpr (SPLIT > 1) cluster_wait();   // no CTA leaves while a peer may read it
    }
}

// ------------------------------------------------------------------ any D <= 256

// One CTA per (sequence, head), one warp per row (rows strided over 4 warps),
// lanes strided over columns with the row cached in registers, so the state is
// still read once and written once.  Handles D < 32, D not a multiple of 32,
// and any element alignment.
constexpr int kGenWarps = 4;
constexpr int kMaxD = 256;

template <typename TS, bool NORM>
__global__ void __launch_bounds__(kGenWarps * 32)
decode_generic(const DecodeParams p)
{
    constexpr int MAXV = kMaxD / 32;
    __shared__ float o_s[kMaxD];
    __shared__ float red[kGenWarps];

    const int D = p.d;
    const int unit = blockIdx.x;
    const int seq = unit / p.nv;
    const int h = unit - seq * p.nv;
    const int g = h % p.nk;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    TS *S = reinterpret_cast<TS *>(p.state) + seq * p.pitch + (int64_t)h * D * D;
    const float *kp = p.k + seq * p.qk_stride + (int64_t)g * D;
    const float *qp = p.q + seq * p.qk_stride + (int64_t)g * D;
    const float *vp = p.v + seq * p.v_stride + (int64_t)h * D;
    const float alpha = p.alpha[seq * p.gb_stride + h];
    const float beta = p.beta[seq * p.gb_stride + h];

    float kreg[MAXV], qreg[MAXV];
    float kq = 0.f;
#pragma unroll
    for (int j = 0; j < MAXV; ++j) {
        const int c = lane + 32 * j;
        kreg[j] = c < D ? kp[c] : 0.f;
        qreg[j] = c < D ? qp[c] : 0.f;
        kq = fmaf(kreg[j], qreg[j], kq);
    }
    kq = group_sum<32>(kq);

    for (int a = warp; a < D; a += kGenWarps) {
        TS *row = S + (int64_t)a * D;
        float s[MAXV];
        float u = 0.f, w = 0.f;
#pragma unroll
        for (int j = 0; j < MAXV; ++j) {
            const int c = lane + 32 * j;
            s[j] = c < D ? to_f32<TS>(row[c]) : 0.f;
            u = fmaf(s[j], kreg[j], u);
            w = fmaf(s[j], qreg[j], w);
        }
        u = group_sum<32>(u);
        w = group_sum<32>(w);
        const float coef = beta * (vp[a] - alpha * u);
        const float oa = (alpha * w + coef * kq) * p.inv_sqrt_d;
#pragma unroll
        for (int j = 0; j < MAXV; ++j) {
            const int c = lane + 32 * j;
            if (c < D) row[c] = from_f32<TS>(fmaf(coef, kreg[j], alpha * s[j]));
        }
        if (lane == 0) o_s[a] = oa;
    }
    __syncthreads();

    if constexpr (!NORM) {
        for (int a = threadIdx.x; a < D; a += kGenWarps * 32)
            p.o[seq * p.o_stride + (int64_t)h * D + a] = o_s[a];
    } else {
        float ss = 0.f;
        for (int a = threadIdx.x; a < D; a += kGenWarps * 32) ss += o_s[a] * o_s[a];
        ss = group_sum<32>(ss);
        if (lane == 0) red[warp] = ss;
        __syncthreads();
        float tot = 0.f;
#pragma unroll
        for (int i = 0; i < kGenWarps; ++i) tot += red[i];
        const float rstd = rsqrtf(tot / (float)D + p.eps);
        const float *zp = p.z + seq * p.z_stride + (int64_t)h * D;
        uint16_t *op = p.out + seq * p.out_stride + (int64_t)h * D;
        for (int a = threadIdx.x; a < D; a += kGenWarps * 32)
            op[a] = bf16_bits_rn(p.gn[a] * o_s[a] * rstd * silu(zp[a]));
    }
}

template <typename TS, bool NORM>
cudaError_t launch_typed(const DecodeParams &p, bool fast, cudaStream_t s)
{
    const unsigned grid = (unsigned)((int64_t)p.batch * p.nv);
    using F = FastShape<TS>;
    if (fast) {
        auto kern = decode_d128<TS, NORM, F::kWarps, F::kBatches, F::kMinBlocks, F::kSplit>;
        if (F::kSplit == 1) {
            kern<<<grid, F::kWarps * 32, 0, s>>>(p);
        } else {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(grid * F::kSplit, 1, 1);
            cfg.blockDim = dim3(F::kWarps * 32, 1, 1);
            cfg.stream = s;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = F::kSplit;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            return cudaLaunchKernelEx(&cfg, kern, p);
        }
    }
    else decode_generic<TS, NORM><<<grid, kGenWarps * 32, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeParams &p, bool f16_state, bool norm, bool fast, cudaStream_t s)
{
    if (f16_state) {
        return norm ? launch_typed<__half, true>(p, fast, s) : launch_typed<__half, false>(p, fast, s);
    }
    return norm ? launch_typed<float, true>(p, fast, s) : launch_typed<float, false>(p, fast, s);
}

}  // namespace gdn
