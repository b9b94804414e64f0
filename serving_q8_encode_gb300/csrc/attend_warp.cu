// Multi-agent decode attention over the shared pool when each kv head has
// only a few query rows: head_dim 64 with up to 16 rows (SmolLM2-1.7B: one
// query head per kv head, up to 16 agents) or head_dim 128 with up to 8
// (Llama-3-8B: one or two agents, 4 GQA heads). Rows go through the score MMA
// in passes of 8 (d = 64) or 4 (d = 128); a group's key and value operands
// are converted once and used by every pass.
//
// PolyKV abstract ("PolyKV: A Shared Asymmetrically-Compressed KV Cache Pool
// for Multi-Agent LLM Inference"): the agents read one compressed pool, keys
// as q8_0 int8 codes with an fp16 scale per 32-element block, values as 3-bit
// Lloyd-Max codes of the FWHT-rotated unit vector with an fp16 norm. The
// output is the same as that of the other attention kernels: scaled
// dot-product attention over the dequantized pool, with the values
// accumulated in the rotated basis and one inverse FWHT per output row in the
// merge kernel.
//
// With a handful of rows there is too little work per pool tile to pay for
// hand-offs between warps, so every warp is an independent flash-decoding
// worker: it walks a contiguous range of (kv-head unit, 32-token group)
// items, streams each group into its own shared-memory ring with 1-D bulk
// copies (one elected lane, one mbarrier per stage), and keeps its softmax
// state and output accumulator in registers. A range that crosses a unit
// boundary writes one partial per piece (slot = unit + warp range), which the
// merge kernel combines (log-sum-exp, one inverse FWHT per row).
//
// Both contractions of a group run as warp-level m16n8k16 tensor-core MMAs
// (fp16 operands, fp32 accumulate) held entirely in registers:
//
//   scores  S^T[(row, block)][token] = Q'[(row, block)][dims] . Kc[token][dims]^T
//           M = 16 (row, q8_0 block) pairs: 8 rows x 2 blocks at d = 64, 4 rows x 4 blocks at d = 128;
//           Q' holds row r's query (fp16, scaled by a power of two per row) in the dims of block b
//           and zero elsewhere, so each accumulator row is one exact per-block dot product and the
//           block scales are applied afterwards; Kc are the int8 codes as exact fp16.
//   values  O^T[dim][row] += V'[dim][token] . P'[token][row]
//           V' = the centroid of the value code (fp16), P' = 2^(logit - max) * ||v|| * w in fp16
//           (w a power of two from the unit's norm maximum, so P' < 2^15).
//
// The K index of both MMAs is permuted so that every operand is thread-local:
// lane (g, t) of the score MMA reads the key row of token 8(g/2) + 2i + g%2
// of n-tile i, bytes [t D/4, (t+1) D/4) of it (one block at d = 128); its
// score accumulator then holds tokens 8t + 2i + {0, 1} of row g, which are
// exactly the probabilities the value MMA's B fragment needs, and the value
// MMA's A fragment needs the codes of tokens 8t .. 8t+7, i.e. bytes
// [3t, 3t+3) of each coordinate's 12-byte code string, decoded two codes at
// a time through a lane-replicated table of fp16 centroid pairs.
//
// Every mbarrier wait is bounded (2 s); on expiry a warp stops, waits
// (bounded) for its copies in flight and sets the pool's status word.
#include <cmath>

#include "polykv_internal.cuh"
#include "tc_ptx.cuh"

namespace polykv {
namespace {

constexpr int kGroup = 32;                 // tokens per work item (one value-code group)
constexpr float kLog2eW = 1.4426950408889634f;
constexpr uint64_t kWaitNs = 2000000000ull;

// NP = row passes: each group's keys and value codes are converted once and used for NP * RP rows
template <int D, int NP>
struct WCfg {
    static constexpr int NB = D / 32;                  // q8_0 blocks per key vector
    static constexpr int KS = D / 16;                  // K-steps of the score MMA
    static constexpr int RP = 16 / NB;                 // query rows per score MMA (one pass)
    static constexpr int ROWS = NP * RP;               // query rows per kv head this configuration takes
    static constexpr int MT = D / 16;                  // M-tiles of the value MMA
    static constexpr int KEY = kGroup * D;             // stage layout (bytes): key codes
    static constexpr int SCL = kGroup * NB * 2;        // block scales
    static constexpr int VCB = D * 12;                 // value-code strings
    static constexpr int NRM = kGroup * 2;             // norms
    static constexpr int STAGE = KEY + SCL + VCB + NRM;
    // two passes hold twice the accumulators and query fragments: fewer, larger-register warps
    static constexpr int WARPS = NP == 2 ? 8 : (D == 64 ? 8 : 12);   // warps per CTA
    static constexpr int STAGES = NP == 2 ? 4 : (D == 64 ? 4 : 3);   // ring depth per warp
    static constexpr int CTAS = NP == 2 ? 1 : (D == 64 ? 2 : 1);     // CTAs per SM
    static constexpr int LUT = 64 * 32 * 4;            // centroid-pair table, one copy per lane
    static constexpr int SMEM = LUT + WARPS * STAGES * STAGE + WARPS * STAGES * 8;
    static_assert(STAGE % 16 == 0 && KEY % 16 == 0 && SCL % 16 == 0 && VCB % 16 == 0, "16-byte bulk copies");
};

struct WParams {
    PoolView p;
    const uint16_t* q;       // [L][A][Hq][D]
    float* ws_acc;           // [slots][R][D]
    float* ws_ml;            // [slots][R][2]
    int64_t n_ctx, tt;
    int ng, nw, A, Hq, G, R;
    float scale_log2;
};

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Four int8 codes (one 32-bit word) as two exact fp16 pairs: 0x64XX is 1024 + XX in fp16, so
// (c ^ 0x80) placed under 0x64 is 1152 + c, and one packed subtraction leaves c.
__device__ __forceinline__ void i8x4_to_h2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t t = w ^ 0x80808080u;
    const uint32_t a = __byte_perm(t, 0x64646464u, 0x4140);
    const uint32_t b = __byte_perm(t, 0x64646464u, 0x4342);
    const __half2 bias = __half2half2(__ushort_as_half((unsigned short)0x6480));   // 1152
    const __half2 ha = __hsub2(*reinterpret_cast<const __half2*>(&a), bias);
    const __half2 hb = __hsub2(*reinterpret_cast<const __half2*>(&b), bias);
    lo = *reinterpret_cast<const uint32_t*>(&ha);
    hi = *reinterpret_cast<const uint32_t*>(&hb);
}

__device__ __forceinline__ float ex2f(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

// byte offset of the pair of codes at bit SH of a 24-bit code field in the lane-replicated table
// (entry e of lane l at (32 e + l) * 4)
template <int SH>
__device__ __forceinline__ uint32_t pair_offset(uint32_t f) {
    if constexpr (SH >= 7) return (f >> (SH - 7)) & (63u << 7);
    else return (f << (7 - SH)) & (63u << 7);
}

// per-unit value scale w = 2^(7 - e), nmax = f * 2^e with f in [0.5, 1): ||v|| * w <= 2^7
__device__ __forceinline__ float value_wscale(float nmax) {
    int en = 0;
    if (nmax > 0.0f) frexpf(nmax, &en);
    return nmax > 0.0f ? ldexpf(1.0f, 7 - en) : 1.0f;
}

template <int D, int NP, bool BF16>
__global__ void __launch_bounds__(32 * WCfg<D, NP>::WARPS, WCfg<D, NP>::CTAS) attend_warp_kernel(const WParams P) {
    using C = WCfg<D, NP>;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;

    // lane-replicated table of centroid pairs: entry e = (C[e & 7], C[e >> 3]) in fp16, lane l's copy of
    // entry e at byte (32 e + l) * 4
    uint32_t* lut = reinterpret_cast<uint32_t*>(smem);
    for (int e = threadIdx.x; e < 64 * 32; e += blockDim.x) {
        const int idx = e >> 5;
        const __half lo = __float2half_rn(centroid_of(idx & 7));
        const __half hi = __float2half_rn(centroid_of(idx >> 3));
        lut[e] = (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
    }
    unsigned char* ring = smem + C::LUT + warp * C::STAGES * C::STAGE;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::LUT + C::WARPS * C::STAGES * C::STAGE) + warp * C::STAGES;
    if (threadIdx.x == 0) abort_flag = 0;
    if (lane == 0)
        for (int s = 0; s < C::STAGES; ++s) tc::mbar_init(tc::smem_u32(&bars[s]), 1);
    tc::mbar_init_fence();
    __syncthreads();
    // the merge may be scheduled now; it waits for this grid's writes before reading them
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // warp ranges are numbered across CTAs first, so that a grid with fewer ranges than warps still
    // spreads them over every SM
    const int64_t gw = (int64_t)warp * gridDim.x + blockIdx.x;
    if (gw >= P.nw) return;
    const int64_t x0 = gw * P.tt / P.nw, x1 = (gw + 1) * P.tt / P.nw;
    const int n = (int)(x1 - x0);
    const int64_t u_first = x0 / P.ng;
    const int64_t u_last = (x1 - 1) / P.ng;
    const uint32_t ring_u = tc::smem_u32(ring);
    const uint32_t lut_u = tc::smem_u32(lut);
    const uint32_t lane4 = 4u * (uint32_t)lane;

    // streaming cursor (lane 0): pointers to the next group's four fields, advanced one group at a time
    int igi = (int)(x0 - u_first * P.ng);
    const int64_t skip = P.p.cap - (int64_t)P.ng * kGroup;   // tokens from a unit's last group to the next unit
    const int64_t tok_first = u_first * P.p.cap + (int64_t)igi * kGroup;
    const int8_t* pk = P.p.kq + tok_first * D;
    const __half* ps = P.p.ks + tok_first * C::NB;
    const uint8_t* pc = P.p.vc + tok_first * (3 * D / 8);
    const __half* pn = P.p.vn + tok_first;
    auto issue_next = [&](int s) {
        const uint32_t dst = ring_u + (uint32_t)(s * C::STAGE);
        const uint32_t bar = tc::smem_u32(&bars[s]);
        tc::mbar_arrive_expect_tx(bar, C::STAGE);
        tc::bulk_g2s(dst, pk, C::KEY, bar);
        tc::bulk_g2s(dst + C::KEY, ps, C::SCL, bar);
        tc::bulk_g2s(dst + C::KEY + C::SCL, pc, C::VCB, bar);
        tc::bulk_g2s(dst + C::KEY + C::SCL + C::VCB, pn, C::NRM, bar);
        pk += kGroup * D;
        ps += kGroup * C::NB;
        pc += C::VCB;
        pn += kGroup;
        if (++igi == P.ng) {
            igi = 0;
            pk += skip * D;
            ps += skip * C::NB;
            pc += skip * (3 * D / 8);
            pn += skip;
        }
    };
    if (lane == 0)
        for (int k = 0; k < C::STAGES && k < n; ++k) issue_next(k);

    // the norm maxima of this warp's units (at most a few), one per lane, fetched while the first copies fly
    const float nm_lane = u_first + lane <= u_last ? P.p.nmax[u_first + lane] : 0.0f;
    __syncwarp();

    // lane roles: score rows m = g and g + 8 are (row g % RP, block g / RP) and (row g % RP, block g / RP + 8 / RP);
    // this lane's key bytes [t D/4, (t+1) D/4) lie in block bt
    const int r_lane = g % C::RP;
    const int b_lo = g / C::RP, b_hi = b_lo + 8 / C::RP;
    const int bt = (t * D / 4) / 32;
    // key row of token 8(g/2) + 2i + g%2 (n-tile i), bytes from t D/4
    const uint32_t koff = (uint32_t)((8 * (g >> 1) + (g & 1)) * D + t * (D / 4));
    // value strings: this lane's 24-bit field is bytes [3t, 3t+3) of each 12-byte string
    const uint32_t vword = (uint32_t)((3 * t) & ~3);
    const uint32_t vsel = (uint32_t)(((3 * t) & 3) | ((((3 * t) & 3) + 1) << 4) | ((((3 * t) & 3) + 2) << 8));
    // scale pair selector (d = 128): blocks b_lo and b_hi of a token's four
    const uint32_t ssel = (b_lo & 1) ? 0x7632u : 0x5410u;
    const int rem = (int)(P.n_ctx - (int64_t)(P.ng - 1) * kGroup);   // valid tokens of a unit's last group

    int64_t unit = u_first;
    int gi = (int)(x0 - u_first * P.ng);
    float m_run[NP], crow[NP], wsc = 1.0f;   // per pass: running maximum, logit scale
    float2 lsum[NP];
    float o[NP][C::MT][4];
    uint32_t qa[NP][C::KS][4];
    bool fresh = true;   // the segment's state must be (re)initialised
    bool aborted = false;
    int k = 0;

    // end of a segment piece: write this warp's partial (the merge kernel combines the unit's pieces)
    auto finish_piece = [&](int64_t u) {
        const int64_t slot = u + gw;   // segment = unit (one row group), piece = this warp's range
        const float iw = 1.0f / wsc;
#pragma unroll
        for (int pp = 0; pp < NP; ++pp) {
            float l = lsum[pp].x + lsum[pp].y;
            l += __shfl_xor_sync(0xffffffffu, l, 1);
            l += __shfl_xor_sync(0xffffffffu, l, 2);
            const int rbase = pp * C::RP;
            if (t == 0 && g < C::RP && rbase + g < P.R)
                reinterpret_cast<float2*>(P.ws_ml)[slot * P.R + rbase + g] = make_float2(m_run[pp], l);
#pragma unroll
            for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int row = 2 * t + h;
                    if (row < C::RP && rbase + row < P.R) {
                        float* dst = P.ws_acc + (slot * P.R + rbase + row) * D + 16 * mt + g;
                        dst[0] = o[pp][mt][h] * iw;
                        dst[8] = o[pp][mt][2 + h] * iw;
                    }
                }
        }
    };

    for (; k < n; ++k) {
        if (fresh) {
            // a new segment: this lane's query dims [t D/4, (t+1) D/4) of row r_lane, scaled by a power of two
            // so that the row's largest magnitude is in [2^14, 2^15), into the score MMA's A fragments
            const int layer = (int)(unit / P.p.H), kvh = (int)(unit - (int64_t)layer * P.p.H);
#pragma unroll
            for (int pp = 0; pp < NP; ++pp) {
                const int rq = pp * C::RP + r_lane;   // this pass's query row of the lane
                float xq[D / 4];
#pragma unroll
                for (int i = 0; i < D / 4; ++i) xq[i] = 0.0f;
                if (rq < P.R) {
                    const int a = rq / P.G, gq = rq - a * P.G;
                    const uint4* src = reinterpret_cast<const uint4*>(
                        P.q + (((int64_t)layer * P.A + a) * P.Hq + kvh * P.G + gq) * D + t * (D / 4));
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        const uint4 w = __ldg(src + c);
                        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            if (BF16) {
                                xq[8 * c + 2 * e] = __uint_as_float(ws[e] << 16);
                                xq[8 * c + 2 * e + 1] = __uint_as_float(ws[e] & 0xFFFF0000u);
                            } else {
                                const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&ws[e]));
                                xq[8 * c + 2 * e] = f.x;
                                xq[8 * c + 2 * e + 1] = f.y;
                            }
                        }
                    }
                }
                float mx = 0.0f;
#pragma unroll
                for (int i = 0; i < D / 4; ++i) mx = fmaxf(mx, fabsf(xq[i]));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                int eq = 0;
                if (mx > 0.0f) frexpf(mx, &eq);
                const float fq = mx > 0.0f ? ldexpf(1.0f, 15 - eq) : 1.0f;
                crow[pp] = P.scale_log2 / fq;
#pragma unroll
                for (int ks = 0; ks < C::KS; ++ks) {
                    const __half2 h01 = __floats2half2_rn(xq[4 * ks] * fq, xq[4 * ks + 1] * fq);
                    const __half2 h23 = __floats2half2_rn(xq[4 * ks + 2] * fq, xq[4 * ks + 3] * fq);
                    const uint32_t u01 = *reinterpret_cast<const uint32_t*>(&h01);
                    const uint32_t u23 = *reinterpret_cast<const uint32_t*>(&h23);
                    qa[pp][ks][0] = b_lo == bt ? u01 : 0u;
                    qa[pp][ks][1] = b_hi == bt ? u01 : 0u;
                    qa[pp][ks][2] = b_lo == bt ? u23 : 0u;
                    qa[pp][ks][3] = b_hi == bt ? u23 : 0u;
                }
            }
            const int64_t ju = unit - u_first;
            const float nm = __shfl_sync(0xffffffffu, nm_lane, (int)(ju & 31));
            wsc = value_wscale(ju < 32 ? nm : P.p.nmax[unit]);
#pragma unroll
            for (int pp = 0; pp < NP; ++pp) {
                m_run[pp] = -INFINITY;
                lsum[pp] = make_float2(0.0f, 0.0f);
#pragma unroll
                for (int mt = 0; mt < C::MT; ++mt) o[pp][mt][0] = o[pp][mt][1] = o[pp][mt][2] = o[pp][mt][3] = 0.0f;
            }
            fresh = false;
        }

        // bounded wait; the outcome is made warp-uniform (and the warp converged) before the MMAs
        const int s = k % C::STAGES;
        const bool ok = tc::mbar_wait(tc::smem_u32(&bars[s]), (uint32_t)((k / C::STAGES) & 1), &abort_flag, kWaitNs);
        if (!__all_sync(0xffffffffu, ok)) {
            aborted = true;
            break;
        }
        const uint32_t st = ring_u + (uint32_t)(s * C::STAGE);

        const bool ragged = gi == P.ng - 1 && rem < kGroup;
        // ---- scores: S^T[(row, block)][token] for tokens 8t + 2i + {0, 1} of this lane's row, n-tile i;
        //      each key fragment is converted once and used by every pass
        float sc[NP][4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
#pragma unroll
            for (int pp = 0; pp < NP; ++pp) sc[pp][i][0] = sc[pp][i][1] = sc[pp][i][2] = sc[pp][i][3] = 0.0f;
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
                const uint4 w = lds128(st + koff + (uint32_t)(2 * i * D + 16 * c));
                const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    uint32_t b0, b1;
                    i8x4_to_h2x2(ws[e], b0, b1);
#pragma unroll
                    for (int pp = 0; pp < NP; ++pp) mma16816(sc[pp][i], qa[pp][4 * c + e], b0, b1);
                }
            }
        }

        // block scales and norms of tokens 8t .. 8t+7 (scales [token][block] fp16, norms [token] fp16)
        float2 s_lo[4], s_hi[4], nw[4];   // per token pair (2i, 2i+1): scale of block b_lo / b_hi, norm * w
        {
            const uint32_t sbase = st + C::KEY + (uint32_t)(t * 8 * C::NB * 2);
            uint32_t sw[8];   // per token: (scale b_lo, scale b_hi) as an fp16 pair
            if constexpr (C::NB == 2) {
                const uint4 a = lds128(sbase), b = lds128(sbase + 16);
                sw[0] = a.x; sw[1] = a.y; sw[2] = a.z; sw[3] = a.w;
                sw[4] = b.x; sw[5] = b.y; sw[6] = b.z; sw[7] = b.w;
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint4 a = lds128(sbase + 16u * c);   // tokens 2c, 2c+1: four scales each
                    sw[2 * c] = __byte_perm(a.x, a.y, ssel);
                    sw[2 * c + 1] = __byte_perm(a.z, a.w, ssel);
                }
            }
            const uint4 nv = lds128(st + C::KEY + C::SCL + C::VCB + (uint32_t)(t * 16));
            const uint32_t nws[4] = {nv.x, nv.y, nv.z, nv.w};
            const __half2 wh = __float2half2_rn(wsc);   // a power of two: exact, and ||v|| w < 2^7
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t plo = __byte_perm(sw[2 * i], sw[2 * i + 1], 0x5410);
                const uint32_t phi = __byte_perm(sw[2 * i], sw[2 * i + 1], 0x7632);
                s_lo[i] = __half22float2(*reinterpret_cast<const __half2*>(&plo));
                s_hi[i] = __half22float2(*reinterpret_cast<const __half2*>(&phi));
                nw[i] = __half22float2(__hmul2(*reinterpret_cast<const __half2*>(&nws[i]), wh));
            }
        }

        if (ragged) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                if (8 * t + 2 * i >= rem) nw[i].x = 0.0f;
                if (8 * t + 2 * i + 1 >= rem) nw[i].y = 0.0f;
            }
        }
        uint32_t pb[NP][4];   // per pass: the value MMA's B fragments
#pragma unroll
        for (int pp = 0; pp < NP; ++pp) {
            // scores with the block scales applied (the row's logit scale is applied with the maximum below)
            float2 y[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                y[i] = __ffma2_rn(s_lo[i], make_float2(sc[pp][i][0], sc[pp][i][1]),
                                  __fmul2_rn(s_hi[i], make_float2(sc[pp][i][2], sc[pp][i][3])));
                if constexpr (C::NB == 4) {   // the other two blocks of the row are in lane g ^ 4
                    y[i].x += __shfl_xor_sync(0xffffffffu, y[i].x, 16);
                    y[i].y += __shfl_xor_sync(0xffffffffu, y[i].y, 16);
                }
            }
            if (ragged) {   // the unit's ragged last group: no weight past n_ctx
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if (8 * t + 2 * i >= rem) y[i].x = -INFINITY;
                    if (8 * t + 2 * i + 1 >= rem) y[i].y = -INFINITY;
                }
            }
            // logits in log2 units relative to the running maximum: y * crow - m
            const float2 cr = make_float2(crow[pp], crow[pp]);
            float2 xl[4];
            {
                const float2 negm = make_float2(-m_run[pp], -m_run[pp]);
#pragma unroll
                for (int i = 0; i < 4; ++i) xl[i] = __ffma2_rn(y[i], cr, negm);
            }
            const float xm = fmaxf(fmaxf(fmaxf(xl[0].x, xl[0].y), fmaxf(xl[1].x, xl[1].y)),
                                   fmaxf(fmaxf(xl[2].x, xl[2].y), fmaxf(xl[3].x, xl[3].y)));
            if (__any_sync(0xffffffffu, xm > 8.0f)) {
                // rare (always on a segment's first group): raise each row's running maximum to at least the
                // group's, rescale what the row has accumulated, and redo the relative logits
                float gm = -INFINITY;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 ya = __fmul2_rn(y[i], cr);
                    gm = fmaxf(gm, fmaxf(ya.x, ya.y));
                }
                gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, 1));
                gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, 2));
                const float m_new = fmaxf(m_run[pp], gm);
                const float alpha = m_run[pp] == -INFINITY ? 0.0f : ex2f(m_run[pp] - m_new);
                m_run[pp] = m_new;
                lsum[pp].x *= alpha;
                lsum[pp].y *= alpha;
                // output rows 2t and 2t+1 of this lane's accumulators take the probabilities of lanes 8t and 8t + 4
                const float a0 = __shfl_sync(0xffffffffu, alpha, 8 * t);
                const float a1 = __shfl_sync(0xffffffffu, alpha, 8 * t + 4);
#pragma unroll
                for (int mt = 0; mt < C::MT; ++mt) {
                    o[pp][mt][0] *= a0;
                    o[pp][mt][1] *= a1;
                    o[pp][mt][2] *= a0;
                    o[pp][mt][3] *= a1;
                }
                const float2 negm = make_float2(-m_run[pp], -m_run[pp]);
#pragma unroll
                for (int i = 0; i < 4; ++i) xl[i] = __ffma2_rn(y[i], cr, negm);
            }

            // probabilities (row sums in fp32) and the value MMA's B fragments P' = p ||v|| w in fp16
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 pr = make_float2(ex2f(xl[i].x), ex2f(xl[i].y));
                lsum[pp] = __fadd2_rn(lsum[pp], pr);
                const float2 pv = __fmul2_rn(pr, nw[i]);
                const __half2 h = __floats2half2_rn(pv.x, pv.y);
                pb[pp][i] = *reinterpret_cast<const uint32_t*>(&h);
            }
        }

        // values: coordinates 16 mt + g and 16 mt + g + 8, tokens 8t .. 8t+7 (k-step j: 8t + 4j + {0, 1, 2, 3});
        // a pair's table offset keeps the lane's byte offset in its low bits
        const uint32_t vbase = st + (uint32_t)(C::KEY + C::SCL) + vword;
#pragma unroll
        for (int mt = 0; mt < C::MT; ++mt) {
            const uint32_t pa = vbase + (uint32_t)((16 * mt + g) * 12);
            const uint32_t fa = __byte_perm(lds32(pa), lds32(pa + 4u), vsel);
            const uint32_t fb = __byte_perm(lds32(pa + 96u), lds32(pa + 100u), vsel);
            uint32_t a[4];
            a[0] = lds32(lut_u + (pair_offset<0>(fa) | lane4));
            a[1] = lds32(lut_u + (pair_offset<0>(fb) | lane4));
            a[2] = lds32(lut_u + (pair_offset<6>(fa) | lane4));
            a[3] = lds32(lut_u + (pair_offset<6>(fb) | lane4));
#pragma unroll
            for (int pp = 0; pp < NP; ++pp) mma16816(o[pp][mt], a, pb[pp][0], pb[pp][1]);
            a[0] = lds32(lut_u + (pair_offset<12>(fa) | lane4));
            a[1] = lds32(lut_u + (pair_offset<12>(fb) | lane4));
            a[2] = lds32(lut_u + (pair_offset<18>(fa) | lane4));
            a[3] = lds32(lut_u + (pair_offset<18>(fb) | lane4));
#pragma unroll
            for (int pp = 0; pp < NP; ++pp) mma16816(o[pp][mt], a, pb[pp][2], pb[pp][3]);
        }

        // release the stage (generic reads ordered before the async-proxy refill) and refill it
        tc::fence_proxy_async();
        __syncwarp();
        if (lane == 0 && k + C::STAGES < n) issue_next(s);

        if (++gi == P.ng) {
            finish_piece(unit);
            ++unit;
            gi = 0;
            fresh = true;
        }
    }
    if (!aborted) {
        if (!fresh) finish_piece(unit);
        return;
    }
    // gave up on a wait: let this warp's copies in flight land (bounded) before the CTA can exit
    const int last = k + C::STAGES < n ? k + C::STAGES : n;
    for (int j = k; j < last; ++j) {
        const uint32_t bar = tc::smem_u32(&bars[j % C::STAGES]);
        const uint32_t par = (uint32_t)((j / C::STAGES) & 1);
        const uint64_t t0 = tc::globaltimer();
        while (!tc::mbar_try(bar, par) && tc::globaltimer() - t0 < 50000000ull) {
        }
    }
    if (lane == 0) atomicOr(P.p.status, 1u);
}

template <int D, int NP>
struct WPlan {
    int64_t ng, tt;
    int nw, nctas;
    size_t slots;
};

template <int D, int NP>
WPlan<D, NP> wplan(const PoolView& p, int64_t n_ctx) {
    using C = WCfg<D, NP>;
    WPlan<D, NP> pl;
    pl.ng = (n_ctx + kGroup - 1) / kGroup;
    pl.tt = (int64_t)p.L * p.H * pl.ng;
    const int64_t warps = (int64_t)device_sm_count() * C::CTAS * C::WARPS;
    pl.nw = (int)(pl.tt < warps ? pl.tt : warps);
    // ranges are numbered across CTAs first (range = warp * grid + CTA): with one CTA per SM slot even
    // a small number of ranges is spread over every SM
    const int64_t slots_ctas = (int64_t)device_sm_count() * C::CTAS;
    pl.nctas = (int)(pl.nw < slots_ctas ? pl.nw : slots_ctas);
    pl.slots = (size_t)((int64_t)p.L * p.H + pl.nw);
    return pl;
}

template <int D, int NP>
size_t warp_workspace(const WPlan<D, NP>& pl, int R) {
    return sizeof(float) * pl.slots * (size_t)R * (size_t)(D + 2);
}

template <int D, int NP, bool BF16>
polykv_status run_warp(const PoolView& p, const void* q, float* out, int A, int Hq, int64_t n_ctx, float scale,
                       void* ws, size_t ws_bytes, cudaStream_t stream, const SuffixArgs* sfx) {
    using C = WCfg<D, NP>;
    const int G = Hq / p.H, R = A * G;
    const WPlan<D, NP> pl = wplan<D, NP>(p, n_ctx);
    const size_t need = warp_workspace<D, NP>(pl, R);
    if (ws_bytes < need) return set_error(POLYKV_E_BUFFER_TOO_SMALL, "attend: workspace %zu < %zu bytes", ws_bytes, need);
    if (pl.ng > 0x7FFFFFFF) return set_error(POLYKV_E_UNSUPPORTED, "attend: context too long");
    WParams P;
    P.p = p;
    P.q = static_cast<const uint16_t*>(q);
    P.ws_acc = static_cast<float*>(ws);
    P.ws_ml = P.ws_acc + pl.slots * (size_t)R * D;
    P.n_ctx = n_ctx;
    P.tt = pl.tt;
    P.ng = (int)pl.ng;
    P.nw = pl.nw;
    P.A = A;
    P.Hq = Hq;
    P.G = G;
    P.R = R;
    P.scale_log2 = scale * kLog2eW;
    auto kern = attend_warp_kernel<D, NP, BF16>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return set_error(POLYKV_E_CUDA, "attend_warp: smem attribute: %s", cudaGetErrorString(e));
    kern<<<pl.nctas, 32 * C::WARPS, C::SMEM, stream>>>(P);
    e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(POLYKV_E_CUDA, "attend_warp launch: %s", cudaGetErrorString(e));
    if (sfx) {
        const polykv_status ss = launch_attend_suffix(*sfx, BF16 ? POLYKV_BF16 : POLYKV_F16, p.L, A, p.H, Hq, D, scale, stream);
        if (ss != POLYKV_OK) return ss;
    }
    MergeLayout ml;
    ml.nrg = 1;
    ml.RS = R;
    ml.nt = pl.ng;
    ml.tt = pl.tt;
    ml.nc = pl.nw;
    return launch_attend_merge(P.ws_acc, P.ws_ml, out, p.L * p.H, p.H, A, Hq, R, 0, ml, D, stream,
                               sfx ? sfx->acc : nullptr, sfx ? sfx->ml : nullptr);
}

}  // namespace

bool attend_warp_supported(const PoolView& p, int rows) {
    return rows >= 1 && ((p.d == 64 && rows <= WCfg<64, 2>::ROWS) || (p.d == 128 && rows <= WCfg<128, 2>::ROWS));
}

size_t attend_warp_workspace(const PoolView& p, int rows, int64_t n_ctx) {
    if (p.d == 64)
        return rows <= WCfg<64, 1>::ROWS ? warp_workspace<64, 1>(wplan<64, 1>(p, n_ctx), rows)
                                         : warp_workspace<64, 2>(wplan<64, 2>(p, n_ctx), rows);
    return rows <= WCfg<128, 1>::ROWS ? warp_workspace<128, 1>(wplan<128, 1>(p, n_ctx), rows)
                                      : warp_workspace<128, 2>(wplan<128, 2>(p, n_ctx), rows);
}

polykv_status launch_attend_warp(const PoolView& p, polykv_dtype dt, const void* q, float* out, int n_agents,
                                 int n_q_heads, int64_t n_ctx, float scale, void* ws, size_t ws_bytes,
                                 cudaStream_t stream, const SuffixArgs* sfx) {
    const int rows = n_agents * (n_q_heads / p.H);
    if (!attend_warp_supported(p, rows))
        return set_error(POLYKV_E_UNSUPPORTED, "warp attend: d=%d rows=%d", p.d, rows);
    const bool bf = dt == POLYKV_BF16;
#define POLYKV_RUN_WARP(D_, NP_)                                                                              \
    return bf ? run_warp<D_, NP_, true>(p, q, out, n_agents, n_q_heads, n_ctx, scale, ws, ws_bytes, stream, sfx) \
              : run_warp<D_, NP_, false>(p, q, out, n_agents, n_q_heads, n_ctx, scale, ws, ws_bytes, stream, sfx)
    if (p.d == 64) {
        if (rows <= WCfg<64, 1>::ROWS) POLYKV_RUN_WARP(64, 1);
        POLYKV_RUN_WARP(64, 2);
    }
    if (rows <= WCfg<128, 1>::ROWS) POLYKV_RUN_WARP(128, 1);
    POLYKV_RUN_WARP(128, 2);
#undef POLYKV_RUN_WARP
}

}  // namespace polykv
