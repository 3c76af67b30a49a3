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
//  * one CTA owns one (sequence, head) -- 8 warps x 16 rows, or 16 warps x 8
//    rows on grids of one wave -- so the norm's reduction over the head's D
//    outputs needs a single __syncthreads;
//  * every state access is a 16-byte vector: an fp32 row (512 B) is one
//    warp-wide load, an fp16 row (256 B) half of one, so a warp touches whole
//    128-byte lines and stores never leave partial sectors;
//  * the whole head is staged in shared memory by cp.async (64 KB fp32,
//    32 KB fp16): each lane issues every 16-byte load of its slice at once,
//    in four commit groups, and computes group g while groups > g land.  The
//    loads hold no registers while in flight, so 3 (fp32) or 4 (fp16) CTAs
//    per SM keep 128-192 KB of reads outstanding per SM -- enough to cover
//    HBM latency at full bandwidth while the stores of earlier rows drain.
//    Each lane reads back only the vectors it copied itself;
//  * k and q are read as this lane's own 16-byte columns, v/z/gn as one
//    coalesced read per warp (a float per row) that lanes broadcast by shuffle;
//  * k.q is a butterfly sum inside the group of lanes that holds a row (32
//    lanes fp32, 16 lanes fp16), once per warp; the rows' u = S[a].k and
//    w = S[a].q are reduced a group of rows at a time (a commit group, a
//    register batch, or all of a lane's rows on one-wave grids) by one
//    transposed butterfly: a reduce-scatter with the butterfly's partners, so
//    every sum keeps the butterfly's bits, in about 2 shuffles a row instead
//    of 8-10 and one chain of levels a group instead of one a row (48-layer
//    step 1.520 -> 1.508 ms, single-layer step 3.20 -> 2.80 us);
//  * on grids of one wave (batch 1-3 at 48 heads), where a step's time is the
//    CTA's own dependency chain rather than HBM, four warps finish the norm,
//    a row per lane, while the rest return.
#include "gdn_internal.cuh"

#ifndef STAGED_MIN_CTAS_PER_SM
#define STAGED_MIN_CTAS_PER_SM 8
#endif
#ifndef DECODE_PATH_FORCE
#define DECODE_PATH_FORCE -1
#endif

namespace gdn {
namespace {

constexpr int kD = 128;

// ------------------------------------------------------------------ D == 128

// Three ways to bring a lane's 16-byte state vectors in, all with the same
// arithmetic (bitwise-identical results).  The staged and register-batched
// paths run 8 warps x 16 rows per head (16 fp32 or 8 fp16 vectors a lane);
// the all-in-registers path runs 16 warps x 8 rows (W = 2 * kWarps: 8 fp32 or
// 4 fp16 vectors a lane, and lanes r < 8 carry the rows' o):
//  * staged: every load in flight at once through cp.async into shared memory
//    (64 KB fp32 / 32 KB fp16 per CTA), four commit groups each consumed as it
//    lands.  The loads hold no registers while in flight, so 3 (fp32) or 4
//    (fp16) CTAs per SM keep 128-192 KB outstanding per SM: for large calls;
//  * register batches (NB > 1): batch b + 1 in flight while batch b is
//    computed, one hop less per element than staging;
//  * all in registers (NB == 1): every load in flight at once, for grids of at
//    most one CTA per SM, where occupancy does not matter.
// The launcher picks one per call (pick_path below).
constexpr int kWarps = 8;
constexpr int kGroups = 4;                     // cp.async commit groups per lane (staged)
template <typename TS> struct StagedShape { static constexpr int kMinBlocks = 3; };
template <> struct StagedShape<__half> { static constexpr int kMinBlocks = 4; };
template <typename TS> struct RegShape { static constexpr int kBatches = 4, kMinBlocks = 3; };   // fp32 only

template <typename TS>
constexpr int stage_bytes() { return kD * kD * (int)sizeof(TS); }

template <typename TS, int EPI, bool STAGED, int NB, int MINB, bool EARLY, int W = kWarps>
__global__ void __launch_bounds__(W * 32, MINB)
decode_d128(const DecodeParams p)
{
    constexpr bool NORM = EPI != kEpiRaw;
    using V = Vec16<TS>;
    constexpr int EPV = V::N;                  // state elements per 16-byte vector
    constexpr int LPR = kD / EPV;              // lanes per state row: 32 fp32, 16 fp16
    constexpr int RPL = 32 / LPR;              // rows per warp-wide access: 1 fp32, 2 fp16
    constexpr int RPW = kD / W;                // rows per warp
    constexpr int NLD = RPW / RPL;             // 16-byte state vectors per lane
    constexpr int VPR = kD * (int)sizeof(TS) / 16;   // vectors per state row
    constexpr int NBAT = STAGED ? kGroups : NB;      // groups / batches of loads
    constexpr int PER = NLD / NBAT;                  // vectors per group / batch
    static_assert(NLD % NBAT == 0 && RPW <= 32, "shape");
    // the one-wave path (every load in registers, at most one CTA per SM): the norm is finished by
    // the first kD / 32 warps, a row per lane, after the barrier
    constexpr bool ONE_WAVE = !STAGED && NB == 1;

    const int unit = blockIdx.x;               // (sequence, value head)
    const int seq = unit / p.nv;
    const int h = unit - seq * p.nv;
    const int g = h % p.nk;                    // tiled key-head pairing
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int sub = lane / LPR;                // which row of a warp-wide access
    const int col = (lane % LPR) * EPV;        // first column this lane owns
    const int row0 = warp * RPW;

    TS *head = reinterpret_cast<TS *>(p.state) + seq * p.pitch + (int64_t)h * kD * kD;
    TS *rowp = head + (int64_t)(row0 + sub) * kD + col;
    early_start<EARLY>(head, p.pf_bytes);

    // 1. the state loads in flight before anything else
    extern __shared__ __align__(16) unsigned char smem_raw[];   // staged: [kD rows][VPR], the head as stored
    uint4 *mine = reinterpret_cast<uint4 *>(smem_raw) + (row0 + sub) * VPR + (lane % LPR);
    uint4 raw[STAGED ? 1 : (NB > 1 ? 2 : 1)][STAGED ? 1 : PER];
    if constexpr (STAGED) {
#pragma unroll
        for (int gi = 0; gi < kGroups; ++gi) {
#pragma unroll
            for (int ii = 0; ii < PER; ++ii) {
                const int i = gi * PER + ii;
                cp_async16(mine + i * RPL * VPR, rowp + (int64_t)i * RPL * kD);
            }
            cp_async_commit();
        }
    } else {
#pragma unroll
        for (int i = 0; i < PER; ++i) raw[0][i] = ld_stream16(rowp + (int64_t)i * RPL * kD);
    }

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
    // z, gn: lane r of every warp for row row0 + r; on the one-wave path the norm's tail runs on the
    // first kD / 32 warps, a row per lane (row 32 warp + lane), so those load the tail's rows instead
    float z_l = 0.f, gn_l = 0.f;
    if (NORM && (ONE_WAVE ? warp < kD / 32 : row_lane)) {
        const int zr = ONE_WAVE ? 32 * warp + lane : row0 + lane;
        z_l = __ldg(p.z + seq * p.z_stride + (int64_t)h * kD + zr);
        gn_l = __ldg(p.gn + zr);
    }
    const float alpha = __ldg(p.alpha + seq * p.gb_stride + h);
    const float beta = __ldg(p.beta + seq * p.gb_stride + h);

    float kq = 0.f;
#pragma unroll
    for (int j = 0; j < EPV; ++j) kq = fmaf(kx[j], qx[j], kq);
    kq = group_sum<LPR>(kq);

    // 3. per row: two dot products, the delta coefficient, output, write-back (in groups of rows)
    float o_keep = 0.f;                        // lane r keeps o of row row0 + r
    float o_sq = 0.f;                          // sum of o^2 over the rows of this lane's row group
    // A group of PER vectors (a commit group, a register batch, or on the one-wave path all of the
    // lane's rows) at once: the partial dot products of its rows, then one reduce-scatter over the row
    // group's lanes (reduce_scatter: the butterfly's sums bit for bit), after which the R = LPR /
    // (2 PER) lanes of block m of the group hold value m: u (m even) or w (m odd) of vector m / 2.
    // About 2 shuffles a row instead of 2 log2(LPR), and one chain of log2(LPR) levels a group
    // instead of one a row (measured at batch 1: ~310 cycles a row, one row after another).
    auto group_step = [&](const uint4 (&vec)[PER], const int i0) {
        constexpr int R = LPR / (2 * PER);
        static_assert(R >= 1, "a group's 2 PER values over the LPR lanes of a row");
        float part[2 * PER];
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            float s[EPV];
            V::unpack(vec[i], s);
            float u = 0.f, w = 0.f;
#pragma unroll
            for (int j = 0; j < EPV; ++j) { u = fmaf(s[j], kx[j], u); w = fmaf(s[j], qx[j], w); }
            part[2 * i] = u;
            part[2 * i + 1] = w;
        }
        const float mine_sum = reduce_scatter<LPR, 2 * PER>(part, lane);
        const float other = __shfl_xor_sync(kFull, mine_sum, R);
        const bool is_w = ((lane % LPR) / R) & 1;
        const float u = is_w ? other : mine_sum, w = is_w ? mine_sum : other;
        const int vi = (lane % LPR) / (2 * R);               // the vector (row) these lanes reduced
        const float va = __shfl_sync(kFull, v_l, (i0 + vi) * RPL + sub);
        const float coef = beta * (va - alpha * u);
        const float oa = (alpha * w + coef * kq) * p.inv_sqrt_d;
        // every lane takes its rows' coefficients (and outputs, for the sum of squares in row order)
        const int gbase = lane & ~(LPR - 1);
        float cf[PER];
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            cf[i] = __shfl_sync(kFull, coef, gbase + 2 * R * i);
            if constexpr (NORM) {
                const float oi = __shfl_sync(kFull, oa, gbase + 2 * R * i);
                o_sq = fmaf(oi, oi, o_sq);
            }
        }
        {   // lane r < RPW keeps the o of row r: vector r / RPL of row group r % RPL
            const int vr = lane / RPL - i0;
            const float ok = __shfl_sync(kFull, oa, (lane % RPL) * LPR + (vr & (PER - 1)) * 2 * R);
            if (lane < RPW && vr >= 0 && vr < PER) o_keep = ok;
        }
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            float s[EPV];
            V::unpack(vec[i], s);
#pragma unroll
            for (int j = 0; j < EPV; ++j) s[j] = fmaf(cf[i], kx[j], alpha * s[j]);
            st_stream16(rowp + (int64_t)(i0 + i) * RPL * kD, V::pack(s));
        }
    };
#pragma unroll
    for (int bt = 0; bt < NBAT; ++bt) {
        if constexpr (STAGED) {
            if (bt == 0) cp_async_wait<kGroups - 1>();
            else if (bt == 1) cp_async_wait<kGroups - 2>();
            else if (bt == 2) cp_async_wait<kGroups - 3>();
            else cp_async_wait<0>();
            uint4 vec[PER];
#pragma unroll
            for (int ii = 0; ii < PER; ++ii) vec[ii] = mine[(bt * PER + ii) * RPL * VPR];
            group_step(vec, bt * PER);
        } else {
            if (bt + 1 < NBAT) {
#pragma unroll
                for (int i = 0; i < PER; ++i)
                    raw[(bt + 1) & 1][i] = ld_stream16(rowp + (int64_t)((bt + 1) * PER + i) * RPL * kD);
            }
            group_step(raw[bt & 1], bt * PER);
        }
    }

    if constexpr (!NORM) {
        if (row_lane) p.o[seq * p.o_stride + (int64_t)h * kD + row0 + lane] = o_keep;
    } else {
        // 4. gated RMS norm over the head's 128 outputs, in this CTA
        __shared__ float red[W];
        // One-wave path (a CTA's own chain is the time there): the head's o goes to shared memory and
        // the first kD / 32 warps finish the head after the barrier, a row per lane, while the others
        // return; they take the gate's silu(z) before the barrier, as the other warps finish their
        // rows.  Measured per single-layer step: fp32 batch 1 2.835 -> 2.811 us, batch 2 3.50 -> 3.18,
        // fp16 batch 1 2.24 -> 2.05.  The HBM-bound paths take silu after the barrier (0.9 % slower
        // before it).  Either way silu is the product's last factor: the same bits.
        __shared__ float o_s[ONE_WAVE ? kD : 1];
        float sz = 0.f;
        if constexpr (ONE_WAVE) {
            if (row_lane) o_s[row0 + lane] = o_keep;
            if (warp < kD / 32) sz = silu(z_l);
        }
        // the warp's sum of squares: each row group's lanes accumulated its rows' o^2 in the loop, so
        // no reduction is left for the tail of the CTA (measured: 48-layer step 1.564 -> 1.517 ms)
        float ss = o_sq;
#pragma unroll
        for (int r = 1; r < RPL; ++r) ss += __shfl_sync(kFull, o_sq, r * LPR);
        if (lane == 0) red[warp] = ss;
        __syncthreads();
        if constexpr (ONE_WAVE) {
            if (warp >= kD / 32) return;       // no barrier follows on this path
        }
        float part[W];                         // pairwise sum of the warps' partials
#pragma unroll
        for (int i = 0; i < W; ++i) part[i] = red[i];
#pragma unroll
        for (int n = W / 2; n >= 1; n /= 2)
#pragma unroll
            for (int i = 0; i < n; ++i) part[i] += part[i + n];
        const float rstd = rsqrtf(part[0] * (1.0f / kD) + p.eps);
        if constexpr (ONE_WAVE) {
            const int row = 32 * warp + lane;
            const float y = gn_l * o_s[row] * rstd * sz;
            if constexpr (EPI == kEpiBf16) {
                p.out[seq * p.out_stride + (int64_t)h * kD + row] = bf16_bits_rn(y);
            } else {                           // this warp's 32 rows are one int8 group
                if (p.y != nullptr) p.y[seq * p.y_stride + (int64_t)h * kD + row] = y;
                float am = fabsf(y);
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) am = fmaxf(am, __shfl_xor_sync(kFull, am, off));
                const float sc = am > 0.f ? am / 127.0f : 1.0f;
                p.xq[seq * p.xq_stride + (int64_t)h * kD + row] = (int8_t)__float2int_rn(y / sc);
                if (lane == 0) p.xs[seq * p.xs_stride + (int64_t)h * (kD / 32) + warp] = sc;
            }
        } else if constexpr (EPI == kEpiBf16) {
            if (row_lane) {
                const float y = gn_l * o_keep * rstd * silu(z_l);
                p.out[seq * p.out_stride + (int64_t)h * kD + row0 + lane] = bf16_bits_rn(y);
            }
        } else {
            // int8 groups of 32: a group is the rows of 32 / RPW consecutive warps.  Each warp takes the
            // max |y| over its rows (lanes r < RPW hold them), the group's warps exchange theirs through
            // shared memory, and every warp quantises its own rows (the same max, the same IEEE division
            // as quant_group32: the same codes).
            constexpr int WPG = 32 / RPW;                   // warps per group
            __shared__ float wmax[W];
            float y = 0.f;
            if (row_lane) {
                y = gn_l * o_keep * rstd * silu(z_l);
                if (p.y != nullptr) p.y[seq * p.y_stride + (int64_t)h * kD + row0 + lane] = y;
            }
            float am = fabsf(y);
#pragma unroll
            for (int off = RPW / 2; off > 0; off >>= 1) am = fmaxf(am, __shfl_xor_sync(kFull, am, off));
            if (lane == 0) wmax[warp] = am;
            __syncthreads();
            const int g0 = warp - warp % WPG;
            float gm = wmax[g0];
#pragma unroll
            for (int i = 1; i < WPG; ++i) gm = fmaxf(gm, wmax[g0 + i]);
            const float sc = gm > 0.f ? gm / 127.0f : 1.0f;
            if (row_lane)
                p.xq[seq * p.xq_stride + (int64_t)h * kD + row0 + lane] = (int8_t)__float2int_rn(y / sc);
            if (warp == g0 && lane == 0) p.xs[seq * p.xs_stride + (int64_t)h * (kD / 32) + row0 / 32] = sc;
        }
    }
}

// ------------------------------------------------------------------ any D <= 256

// One CTA per (sequence, head), one warp per row (rows strided over 4 warps),
// lanes strided over columns with the row cached in registers, so the state is
// still read once and written once.  Handles D < 32, D not a multiple of 32,
// and any element alignment.
constexpr int kGenWarps = 4;
constexpr int kMaxD = 256;

template <typename TS, int EPI, bool EARLY>
__global__ void __launch_bounds__(kGenWarps * 32)
decode_generic(const DecodeParams p)
{
    constexpr bool NORM = EPI != kEpiRaw;
    constexpr int MAXV = kMaxD / 32;
    __shared__ float o_s[kMaxD];
    __shared__ float red[kGenWarps];
    early_start<EARLY>(nullptr, 0);            // no prefetch: rows need not be aligned here

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
        for (int a = threadIdx.x; a < D; a += kGenWarps * 32) {
            const float y = p.gn[a] * o_s[a] * rstd * silu(zp[a]);
            if constexpr (EPI == kEpiBf16) {
                p.out[seq * p.out_stride + (int64_t)h * D + a] = bf16_bits_rn(y);
            } else {
                o_s[a] = y;                    // this thread's own entry
                if (p.y != nullptr) p.y[seq * p.y_stride + (int64_t)h * D + a] = y;
            }
        }
        if constexpr (EPI == kEpiQ8) {        // D % 32 == 0 (checked on the host)
            __syncthreads();
            for (int grp = warp; grp < D / 32; grp += kGenWarps)
                quant_group32(o_s[32 * grp + lane], p.xq + seq * p.xq_stride + (int64_t)h * D + 32 * grp + lane,
                              p.xs + seq * p.xs_stride + (int64_t)h * (D / 32) + grp, lane);
        }
    }
}

// Which of the D == 128 variants a call takes, from per-launch times measured
// on GB300 for batch 1..32 (NV = 48), fp32 and fp16, with the state in L2 (one
// layer repeated) and streaming from HBM (48 distinct layers):
//  * grid <= one CTA per SM (latency-bound, occupancy moot): every load of a
//    lane in flight at once, in registers.  Best for fp16 in both cases; for
//    fp32 within 8 % of the best in both (register batches are 8 % faster from
//    L2 but 11 % slower from HBM, staging the reverse);
//  * fp32 up to kStagedMinCtasPerSm CTAs per SM: register batches;
//  * otherwise staged.
enum class Path { kRegAll, kRegBatched, kStaged };
constexpr int kStagedMinCtasPerSm = STAGED_MIN_CTAS_PER_SM;

template <typename TS>
Path pick_path(unsigned grid)
{
#if DECODE_PATH_FORCE >= 0
    (void)grid;
    return static_cast<Path>(DECODE_PATH_FORCE);
#else
    const unsigned sms = (unsigned)sm_count();
    if (grid <= sms) return Path::kRegAll;
    if (sizeof(TS) == 4 && grid < (unsigned)kStagedMinCtasPerSm * sms) return Path::kRegBatched;
    return Path::kStaged;
#endif
}

template <typename TS, int EPI>
cudaError_t launch_typed(const DecodeParams &p, bool fast, cudaStream_t s)
{
    const unsigned grid = (unsigned)((int64_t)p.batch * p.nv);
    if (!fast) {
        if (grid <= (unsigned)sm_count())      // one wave: launched early (the tiny-config chain)
            return launch_early(decode_generic<TS, EPI, true>, grid, kGenWarps * 32, 0, s, true, p);
        decode_generic<TS, EPI, false><<<grid, kGenWarps * 32, 0, s>>>(p);
        return cudaGetLastError();
    }
    // Early launch (grids of a few waves, see early_grid) with the first sixteenth of the head asked
    // of the L2.  More is faster on its own but slower when host copies run beside the kernels:
    // 48-layer step at batch 32, device-only / with per-layer host copies on a second stream, ms:
    // a quarter 1.491 / 1.561, an eighth 1.501 / 1.544, a sixteenth 1.508 / 1.537, none 1.515 /
    // 1.535 (with rows reduced one at a time a quarter had been best: 1.520 / 1.551).
    DecodeParams q = p;
    q.pf_bytes = (unsigned)(kD * kD * sizeof(TS) / 16);
    static_assert(kStagedMinCtasPerSm <= kEarlyMaxWaves * RegShape<float>::kMinBlocks,
                  "register-batched grids must stay within the early-launch waves");
    switch (pick_path<TS>(grid)) {
    case Path::kRegAll:                          // one wave at most: 16 warps x 8 rows a CTA
        return launch_early(decode_d128<TS, EPI, false, 1, 1, true, 2 * kWarps>, grid, 2 * kWarps * 32, 0, s,
                            true, q);
    case Path::kRegBatched:                      // under kStagedMinCtasPerSm / 3 waves
        if constexpr (sizeof(TS) == 4)
            return launch_early(decode_d128<TS, EPI, false, RegShape<TS>::kBatches, RegShape<TS>::kMinBlocks, true>,
                                grid, kWarps * 32, 0, s, true, q);
        [[fallthrough]];
    default: {
        constexpr int M = StagedShape<TS>::kMinBlocks;
        if (early_grid(grid, M)) {
            constexpr auto kern = decode_d128<TS, EPI, true, 1, M, true>;
            const cudaError_t e = allow_dynamic_smem<kern>(stage_bytes<TS>());
            if (e != cudaSuccess) return e;
            return launch_early(kern, grid, kWarps * 32, stage_bytes<TS>(), s, true, q);
        }
        constexpr auto kern = decode_d128<TS, EPI, true, 1, M, false>;
        const cudaError_t e = allow_dynamic_smem<kern>(stage_bytes<TS>());
        if (e != cudaSuccess) return e;
        return launch_early(kern, grid, kWarps * 32, stage_bytes<TS>(), s, false, p);
    }
    }
}

}  // namespace

cudaError_t launch_decode(const DecodeParams &p, bool f16_state, int epi, bool fast, cudaStream_t s)
{
    if (f16_state) {
        switch (epi) {
        case kEpiRaw: return launch_typed<__half, kEpiRaw>(p, fast, s);
        case kEpiBf16: return launch_typed<__half, kEpiBf16>(p, fast, s);
        default: return launch_typed<__half, kEpiQ8>(p, fast, s);
        }
    }
    switch (epi) {
    case kEpiRaw: return launch_typed<float, kEpiRaw>(p, fast, s);
    case kEpiBf16: return launch_typed<float, kEpiBf16>(p, fast, s);
    default: return launch_typed<float, kEpiQ8>(p, fast, s);
    }
}

}  // namespace gdn
