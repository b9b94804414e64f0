// Multi-agent decode attention over the shared pool on the 5th-generation
// tensor cores (tcgen05, TMEM accumulators), head_dim 128, any number of
// query rows per kv head (agents x GQA group), taken in row groups of 64.
//
// PolyKV abstract ("PolyKV: A Shared Asymmetrically-Compressed KV Cache Pool
// for Multi-Agent LLM Inference"): N agents read one compressed pool. With 15
// agents x 4 GQA heads = 60 rows per kv head, q.K and p.V are dense
// contractions (about 156 flop per pool byte), so both run as tcgen05.mma:
//
//   MMA1 (per 128-token tile): S^T[token][row] = K_hat[token][128] . Q'[row][128]^T
//        with K_hat = s_b * code * 2^-4 split exactly into two fp16 halves
//        (hi = fp16(K_hat), lo = K_hat - hi; the product has at most 18
//        significant bits, so hi + lo = K_hat) held in TMEM as the A operand,
//        and Q' the rows' queries in fp16 scaled by a power of two (bf16
//        queries are then exact). One fp32 accumulator sums hi then lo.
//   softmax (one thread per token and row group; TMEM lane = token):
//        d = c * S - m (base-2 logits relative to the running max), lazy
//        rescaling only when some d exceeds 2^8 (decided for the whole row
//        group with one OR-reducing barrier), p = 2^d stored as fp16.
//   MMA2: O^T[dim][row] += Vn[token][dim]^T . P[token][row], where
//        Vn = centroid(code) * ||v|| * w in fp16 (w a power of two from the
//        pool's per-unit norm maximum, so ||v|| w < 2^8): the value operand
//        carries its norm, in the ROTATED basis; the merge kernel applies the
//        inverse FWHT once per output row.
//
// Data movement: one TMA thread streams each tile's block scales, value codes
// and norms (7.25 KB) into a 4-deep shared-memory ring; the key-code rows
// (16 KB per tile) are copied by the producer warps themselves with cp.async,
// one own tile ahead, into padded per-token rows. The ring's readers fence
// the async proxy before releasing a stage (the TMA refill is an async-proxy
// write after their generic loads). Every pool byte is read from HBM
// once for all agents of a row group. A segment is one (layer, kv head, row
// group); the (segment, tile) list is cut into one contiguous range per CTA
// (one persistent CTA per SM), a range that crosses a segment boundary writes
// one softmax partial per segment piece, and the merge kernel combines them.
//
// Warp roles (832 threads): 0-7 producers in two groups of four warps that
// take alternate tiles (each thread: one token's key codes -> exact hi/lo fp16
// in TMEM, then its value codes -> norm-scaled centroids in shared memory),
// 8-23 softmax in four row groups of 16 (one warp per TMEM lane quadrant and
// group), 24 MMA issue (an event loop over both MMA chains, run by the whole
// warp with one elected lane issuing) + TMEM owner, 25 TMA. Every mbarrier
// wait is bounded (2 s); on expiry the CTA raises an abort flag, skips the
// rest of its work, waits (bounded) for its copies in flight, frees its TMEM
// and sets the pool's status word.
#include <cmath>
#include <cstdlib>
#include <cstring>

#include "polykv_internal.cuh"
#include "tc_ptx.cuh"

namespace polykv {
namespace {

constexpr int kTile = 128;
constexpr int kD = 128;
constexpr int kNR = 64;            // padded rows (MMA N)
constexpr int kGroups = 4;                       // softmax row groups
constexpr int kGRows = kNR / kGroups;            // 16 query rows per group
constexpr int kSmWarps = 4 * kGroups;            // softmax warps (one per TMEM lane quadrant and group)
constexpr int kSmThreads = 32 * kSmWarps;
constexpr int kWarpMma = 8 + kSmWarps;           // MMA issue + TMEM owner
constexpr int kWarpTma = kWarpMma + 1;
constexpr int kThreadsTc = 32 * (kWarpTma + 1);  // 26 warps
// named barriers: 1..4 sync one row group, 5..8 OR-reduce within one (never mixed on an id), 9 all softmax
constexpr uint32_t kBarGroup = 1, kBarRed = 5, kBarSoftmax = 9;
constexpr int kNS = 4;             // ring depth: scales / value codes / norms
constexpr int kKS = 4;             // key-row stages: two per producer group (cp.async, one own tile ahead)
constexpr float kTau = 8.0f;       // lazy rescale threshold (log2 units): p <= 2^8
constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr float kLog2eTc = 1.4426950408889634f;

// one ring stage: block scales | value codes | norms
constexpr uint32_t kRawS = 0, kRawV = 1024, kRawN = 7168;
constexpr uint32_t kRawBytes = 7424;       // bytes delivered per tile
constexpr uint32_t kRawStage = 7424;
constexpr uint32_t kKRow = 144;            // padded key row: 8-lane phases of 16-byte loads hit distinct banks
constexpr uint32_t kKStage = kTile * kKRow;

// shared memory map (bytes from a 1024-aligned base)
constexpr uint32_t kSmQ = 0;                            // 2 chunks x [64 rows][128 B]             16 KB
constexpr uint32_t kSmV = kSmQ + 16384;                 // 2 stages x 2 dim blocks x [128][128 B]  64 KB
constexpr uint32_t kSmP = kSmV + 65536;                 // 2 stages x [128 tokens][128 B]          32 KB
constexpr uint32_t kSmRaw = kSmP + 32768;               // kNS x 7.25 KB                           29 KB
constexpr uint32_t kSmK = kSmRaw + kNS * kRawStage;     // kKS x 128 x 144 B                       72 KB
constexpr uint32_t kSmLut = kSmK + kKS * kKStage;       // 64 code pairs x 32 lanes x 4 B            8 KB
constexpr uint32_t kSmMisc = kSmLut + 8192;
constexpr uint32_t kSmBytes = kSmMisc + 3072 + 1024;    // + alignment slack
static_assert(kSmBytes <= 232448, "shared memory budget");
static_assert(kSmK % 16 == 0 && kKRow % 16 == 0, "cp.async destinations are 16-byte aligned");

// TMEM columns
constexpr uint32_t kColK = 0;     // 2 stages x (64 hi + 64 lo)
constexpr uint32_t kColS = 256;   // 2 buffers x 64
constexpr uint32_t kColO = 384;   // 64
constexpr uint32_t kColL = 448;   // 64: per-token-slot partial row sums (lane = token slot)
constexpr uint32_t kTmemCols = 512;

struct TcParams {
    PoolView p;
    const uint16_t* q;
    float* ws_acc;
    float* ws_ml;
    int64_t n_ctx;
    int64_t total_tiles;
    int A, Hq, G;
    int Rtot;    // query rows per kv head (agents x GQA group)
    int nrg;     // groups of up to 64 rows per kv head; a segment is one (kv-head unit, row group)
    int RS;      // rows per partial slot (64 with several row groups, else Rtot)
    int nt;      // tiles per segment (= per unit)
    int nctas;
    int test_stall;  // test hook: the MMA thread issues nothing, so the softmax waits run out
    float scale_log2;
};

struct Misc {
    float m[kNR];         // running max per row (log2 units); +inf for padding rows
    float nm[kNR];        // -m
    float alpha[kNR];     // 2^(m_old - m_new)
    float red[kGroups][4][kGRows];   // per (group, lane quadrant, row): partial maxima or row sums
    float qred[kSmWarps];
    float scale_eff;
    float wscale;
    int abort;
    int pad;
    uint64_t kfull[2], kfree[2], vfull[2], pfull[2], pvfree[2], sfull[2], sfree[2], qready, done;
    uint64_t rfull[kNS], rempty[kNS];
    uint32_t tslot;
};
static_assert(sizeof(Misc) <= 3072, "misc block");

__device__ __forceinline__ int64_t cta_of_tile(int64_t g, int64_t tt, int nc) { return ((g + 1) * nc - 1) / tt; }

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint64_t f2u(float2 a) {
    uint64_t u;
    memcpy(&u, &a, 8);
    return u;
}
__device__ __forceinline__ float2 u2f(uint64_t u) {
    float2 a;
    memcpy(&a, &u, 8);
    return a;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f2u(a)), "l"(f2u(b)));
    return u2f(d);
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f2u(a)), "l"(f2u(b)));
    return u2f(d);
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(f2u(a)), "l"(f2u(b)), "l"(f2u(c)));
    return u2f(d);
}

// OR of `pred` over the `n` threads of named barrier `id`, which all wait here.
__device__ __forceinline__ bool bar_any(uint32_t id, uint32_t n, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n barrier.cta.red.or.pred q, %2, %3, p;\n"
        " selp.u32 %0, 1, 0, q;\n}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}

// 16-byte shared store as inline asm: it stays ahead of the proxy fence and the mbarrier arrive
// that publish it to the tensor cores (a plain store through a restrict pointer could be moved
// past them).
__device__ __forceinline__ void st_shared16(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// 16-byte global -> shared copy, zero-filled when src_bytes == 0
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// int8 x4 -> two fp16x2 words, exactly: fp16(0x6400 | (x ^ 0x80)) = 1024 + x + 128.
__device__ __forceinline__ void i8x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t u = w ^ 0x80808080u;
    const uint32_t magic = 0x64646464u;
    uint32_t a, b;
    asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(a) : "r"(u), "r"(magic));
    asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(b) : "r"(u), "r"(magic));
    const __half2 bias = __half2half2(__ushort_as_half((unsigned short)0x6480));  // 1152
    const __half2 ha = __hsub2(*reinterpret_cast<const __half2*>(&a), bias);
    const __half2 hb = __hsub2(*reinterpret_cast<const __half2*>(&b), bias);
    lo = *reinterpret_cast<const uint32_t*>(&ha);
    hi = *reinterpret_cast<const uint32_t*>(&hb);
}

template <int K>
__device__ __forceinline__ uint32_t code_pair(const uint32_t (&w)[12]) {
    // 6-bit field (two consecutive 3-bit codes) at bit 6K of the 384-bit row
    constexpr int bit = 6 * K, word = bit >> 5, off = bit & 31;
    if constexpr (off <= 26) {
        return (w[word] >> off) & 63u;
    } else {
        return ((w[word] >> off) | (w[word + 1] << (32 - off))) & 63u;
    }
}

// Four 16-byte chunks (dims 8C..8C+31) of one token's value row: centroid pairs looked up
// (all sixteen issued before the stores) and scaled by the token's ||v|| * w.
template <int C>
__device__ __forceinline__ void store_v_quad(const uint32_t (&w)[12], const uint32_t* lut, uint32_t vstage,
                                             uint32_t tok, __half2 nw2) {
    uint32_t o[16];
#define PKV_LUT(I) o[I] = lut[code_pair<4 * C + I>(w) * 32];
    PKV_LUT(0) PKV_LUT(1) PKV_LUT(2) PKV_LUT(3) PKV_LUT(4) PKV_LUT(5) PKV_LUT(6) PKV_LUT(7)
    PKV_LUT(8) PKV_LUT(9) PKV_LUT(10) PKV_LUT(11) PKV_LUT(12) PKV_LUT(13) PKV_LUT(14) PKV_LUT(15)
#undef PKV_LUT
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const __half2 h = __hmul2(*reinterpret_cast<const __half2*>(&o[i]), nw2);
        o[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
#pragma unroll
    for (int q = 0; q < 4; ++q)
        st_shared16(vstage + ((C + q) / 8) * 16384 + tc::sw128(tok, ((C + q) % 8) * 16), o[4 * q], o[4 * q + 1],
                    o[4 * q + 2], o[4 * q + 3]);
}

// Row maxima (in M.red, relative to the running max for a rescale, absolute on a segment's
// first tile) -> new running max and alpha per row of this group. With `scale_o`, O and
// the per-slot row sums are scaled by alpha once MMA2 of the previous tile is done.
__device__ __noinline__ void softmax_new_max(Misc& M, int grp, int tt, int rbase, int R, uint32_t gbar,
                                             bool seg_first, int64_t j, uint32_t lane_addr, volatile int* abortp) {
    tc::named_bar(gbar, 128);
    if (tt < kGRows) {
        const int r = rbase + tt;
        const float mt = fmaxf(fmaxf(M.red[grp][0][tt], M.red[grp][1][tt]),
                               fmaxf(M.red[grp][2][tt], M.red[grp][3][tt]));
        if (seg_first) {
            const float mn = r < R ? mt : INFINITY;
            M.m[r] = mn;
            M.nm[r] = -mn;
            M.alpha[r] = 1.0f;
        } else if (r < R && mt > 0.0f) {
            const float mn = M.m[r] + mt;
            M.alpha[r] = ex2(M.m[r] - mn);
            M.m[r] = mn;
            M.nm[r] = -mn;
        } else {
            M.alpha[r] = 1.0f;
        }
    }
    tc::named_bar(gbar, 128);
    if (!seg_first) {
        // O must be scaled before MMA2 of this tile adds to it
        tc::mbar_wait(tc::smem_u32(&M.pvfree[(j - 1) & 1]), (uint32_t)(((j - 1) >> 1) & 1), abortp, kTimeoutNs);
        tc::fence_after();
#pragma unroll
        for (int cc = 0; cc < kGRows / 16; ++cc) {
            uint32_t to[16], tl[16];
            tc::tmem_ld16(lane_addr + kColO + rbase + 16u * cc, to);
            tc::tmem_ld16(lane_addr + kColL + rbase + 16u * cc, tl);
            tc::wait_ld();
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const float a = M.alpha[rbase + 16 * cc + k];
                to[k] = __float_as_uint(__uint_as_float(to[k]) * a);
                tl[k] = __float_as_uint(__uint_as_float(tl[k]) * a);
            }
            tc::tmem_st16(lane_addr + kColO + rbase + 16u * cc, to);
            tc::tmem_st16(lane_addr + kColL + rbase + 16u * cc, tl);
        }
        tc::wait_st();
    }
}

// per-segment value scale w = 2^(8 - e), nmax = f * 2^e with f in [0.5, 1): ||v|| * w < 2^8
__device__ __forceinline__ float unit_wscale(float nmax) {
    int en = 0;
    if (nmax > 0.0f) frexpf(nmax, &en);
    return nmax > 0.0f ? ldexpf(1.0f, 8 - en) : 1.0f;
}

// Segment prologue (all row groups, every softmax thread): the unit's queries in fp16 scaled by a power
// of two into the MMA1 operand, the logit scale and the value scale w.
template <bool QBF16>
__device__ __noinline__ void softmax_prologue(const uint16_t* __restrict__ q, const float* __restrict__ nmax, int64_t u,
                                              int r0, int H, int A, int Hq, int G, int R, float scale_log2,
                                              uint8_t* sQ, Misc& M, int si, int wi, int lane) {
    const int layer = (int)(u / H), kvh = (int)(u % H);
    uint4 qv[1024 / kSmThreads];
    float qm = 0.0f;
#pragma unroll
    for (int m = 0; m < 1024 / kSmThreads; ++m) {
        const int cid = si + kSmThreads * m;
        qv[m] = make_uint4(0u, 0u, 0u, 0u);
        if (cid < R * 16) {
            const int r = cid >> 4, dc = cid & 15;
            const int a = (r0 + r) / G, gq = (r0 + r) % G;
            qv[m] = __ldg(reinterpret_cast<const uint4*>(
                              q + (((int64_t)layer * A + a) * Hq + kvh * G + gq) * kD) + dc);
            const uint32_t wv[4] = {qv[m].x, qv[m].y, qv[m].z, qv[m].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float lo, hi;
                if (QBF16) {
                    lo = __uint_as_float(wv[e] << 16);
                    hi = __uint_as_float(wv[e] & 0xFFFF0000u);
                } else {
                    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&wv[e]));
                    lo = f.x;
                    hi = f.y;
                }
                qm = fmaxf(qm, fmaxf(fabsf(lo), fabsf(hi)));
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) qm = fmaxf(qm, __shfl_xor_sync(0xffffffffu, qm, o));
    if (lane == 0) M.qred[wi] = qm;
    tc::named_bar(kBarSoftmax, kSmThreads);
    float qmax = 0.0f;
#pragma unroll
    for (int w8 = 0; w8 < kSmWarps; ++w8) qmax = fmaxf(qmax, M.qred[w8]);
    int eq = 0;
    if (qmax > 0.0f) frexpf(qmax, &eq);
    const float fq = qmax > 0.0f ? ldexpf(1.0f, 15 - eq) : 1.0f;  // qmax * fq in [2^14, 2^15)
#pragma unroll
    for (int m = 0; m < 1024 / kSmThreads; ++m) {
        const int cid = si + kSmThreads * m;
        if (cid < kNR * 16) {
            const int r = cid >> 4, dc = cid & 15;
            const uint32_t wv[4] = {qv[m].x, qv[m].y, qv[m].z, qv[m].w};
            uint32_t hv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float lo = 0.0f, hi = 0.0f;
                if (r < R) {
                    if (QBF16) {
                        lo = __uint_as_float(wv[e] << 16);
                        hi = __uint_as_float(wv[e] & 0xFFFF0000u);
                    } else {
                        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&wv[e]));
                        lo = f.x;
                        hi = f.y;
                    }
                }
                const __half2 h = __floats2half2_rn(lo * fq, hi * fq);
                hv[e] = *reinterpret_cast<const uint32_t*>(&h);
            }
            st_shared16(tc::smem_u32(sQ) + (dc >> 3) * 8192 + tc::sw128(r, (dc & 7) * 16), hv[0], hv[1], hv[2], hv[3]);
        }
    }
    if (si == 0) {
        M.scale_eff = scale_log2 * 16.0f / fq;  // keys are stored in TMEM as s * code * 2^-4
        M.wscale = unit_wscale(nmax[u]);
    }
    tc::fence_proxy_async();
    tc::named_bar(kBarSoftmax, kSmThreads);
    if (si == 0) tc::mbar_arrive(tc::smem_u32(&M.qready));
}

// Segment epilogue (one row group): row sums over the token slots, then the rows' O^T columns
// (divided by w) and (m, l) written as the partial for (unit, piece) `slot`.
__device__ __noinline__ void softmax_epilogue(Misc& M, int s, uint32_t ph, volatile int* abortp, uint32_t lane_addr,
                                              int grp, int wq, int lane, int tt, int rbase, int R, int RS,
                                              uint32_t gbar, int64_t slot, float* __restrict__ ws_acc,
                                              float* __restrict__ ws_ml) {
    tc::mbar_wait(tc::smem_u32(&M.pvfree[s]), ph, abortp, kTimeoutNs);
    tc::fence_after();
    tc::wait_st();
#pragma unroll
    for (int cc = 0; cc < kGRows / 16; ++cc) {
        uint32_t tl[16];
        tc::tmem_ld16(lane_addr + kColL + rbase + 16u * cc, tl);
        tc::wait_ld();
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            float v = __uint_as_float(tl[k]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            if (lane == 16 * cc + k) M.red[grp][wq][16 * cc + k] = v;
        }
    }
    tc::named_bar(gbar, 128);
    const float unscale = 1.0f / M.wscale;
#pragma unroll
    for (int cc = 0; cc < kGRows / 16; ++cc) {
        uint32_t to[16];
        tc::tmem_ld16(lane_addr + kColO + rbase + 16u * cc, to);
        tc::wait_ld();
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const int r = rbase + 16 * cc + k;
            if (r < R) ws_acc[(slot * RS + r) * kD + tt] = __uint_as_float(to[k]) * unscale;
        }
    }
    if (tt < kGRows && rbase + tt < R) {
        const int r = rbase + tt;
        ws_ml[(slot * RS + r) * 2] = M.m[r];
        ws_ml[(slot * RS + r) * 2 + 1] =
            M.red[grp][0][tt] + M.red[grp][1][tt] + M.red[grp][2][tt] + M.red[grp][3][tt];
    }
    tc::fence_before();
    tc::named_bar(kBarSoftmax, kSmThreads);
}

template <bool QBF16>
__global__ void __launch_bounds__(kThreadsTc, 1)
    attend_tc_kernel(const TcParams P) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u = tc::smem_u32(smem_raw);
    uint8_t* sm = smem_raw + (((raw_u + 1023u) & ~1023u) - raw_u);
    uint8_t* sQ = sm + kSmQ;
    uint8_t* sV = sm + kSmV;
    uint8_t* sP = sm + kSmP;
    uint8_t* sR = sm + kSmRaw;
    uint8_t* sK = sm + kSmK;
    uint32_t* lut = reinterpret_cast<uint32_t*>(sm + kSmLut);
    Misc& M = *reinterpret_cast<Misc*>(sm + kSmMisc);
    volatile int* abortp = &M.abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t TT = P.total_tiles;
    const int c = blockIdx.x;
    const int64_t g0 = (int64_t)c * TT / P.nctas;
    const int64_t g1 = (int64_t)(c + 1) * TT / P.nctas;
    const int n = (int)(g1 - g0);
    const int nt = P.nt;
    const int64_t cap = P.p.cap;

    // ---- set-up: barriers, codebook pairs, TMEM
    if (tid == 0) {
        for (int s = 0; s < 2; ++s) {
            tc::mbar_init(tc::smem_u32(&M.kfull[s]), 128);
            tc::mbar_init(tc::smem_u32(&M.kfree[s]), 1);
            tc::mbar_init(tc::smem_u32(&M.vfull[s]), 128);
            tc::mbar_init(tc::smem_u32(&M.pfull[s]), kSmThreads);
            tc::mbar_init(tc::smem_u32(&M.pvfree[s]), 1);
            tc::mbar_init(tc::smem_u32(&M.sfull[s]), 1);
            tc::mbar_init(tc::smem_u32(&M.sfree[s]), kSmThreads);
        }
        for (int s = 0; s < kNS; ++s) {
            tc::mbar_init(tc::smem_u32(&M.rfull[s]), 1);
            tc::mbar_init(tc::smem_u32(&M.rempty[s]), 128);
        }
        tc::mbar_init(tc::smem_u32(&M.qready), 1);
        tc::mbar_init(tc::smem_u32(&M.done), 1);
        M.abort = 0;
        tc::mbar_init_fence();
    }
    for (int e = tid; e < 64 * 32; e += kThreadsTc) {
        const int idx = e >> 5;
        const __half lo = __float2half_rn(centroid_of(idx & 7));
        const __half hi = __float2half_rn(centroid_of(idx >> 3));
        lut[e] = (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
    }
    if (warp == kWarpMma) tc::tmem_alloc(tc::smem_u32(&M.tslot), kTmemCols);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tbase = M.tslot;

    if (warp == kWarpTma) {
        // =============================== TMA: scales / value codes / norms into the ring
        if (lane == 0) {
            int issued = 0;
            int64_t sg = g0 / nt;                  // segment
            int64_t u = sg / P.nrg;                // its pool unit
            int ti = (int)(g0 - sg * nt);
            for (int j = 0; j < n && !*abortp; ++j) {
                const int st = j & (kNS - 1);
                if (j >= kNS &&
                    !tc::mbar_wait(tc::smem_u32(&M.rempty[st]), (uint32_t)(((j / kNS) - 1) & 1), abortp, kTimeoutNs))
                    break;
                const int64_t row0 = u * cap + (int64_t)ti * kTile;
                if (++ti == nt) {
                    ti = 0;
                    u = ++sg / P.nrg;
                }
                const uint32_t dst = tc::smem_u32(sR + st * kRawStage);
                const uint32_t bar = tc::smem_u32(&M.rfull[st]);
                tc::mbar_arrive_expect_tx(bar, kRawBytes);
                tc::bulk_g2s(dst + kRawS, P.p.ks + row0 * (kD / kQ8Block), 1024, bar);
                tc::bulk_g2s(dst + kRawV, P.p.vc + row0 * (3 * kD / 8), 6144, bar);
                tc::bulk_g2s(dst + kRawN, P.p.vn + row0, 256, bar);
                issued = j + 1;
            }
            // drain: never leave copies in flight into shared memory that is about to be released
            for (int j = issued > kNS ? issued - kNS : 0; j < issued; ++j) {
                volatile int dummy = 0;
                tc::mbar_wait(tc::smem_u32(&M.rfull[j & (kNS - 1)]), (uint32_t)((j / kNS) & 1), &dummy, 50000000ull);
            }
        }
    } else if (warp < 8) {
        // =============================== producers: two groups of four warps take alternate tiles
        // (group pg: tiles pg, pg + 2, ...; TMEM/shared stage pg). Each thread owns one token slot
        // (= TMEM lane) and writes that token's exact key halves to TMEM, then its norm-scaled value
        // centroids to shared memory.
        const int pg = warp >> 2;
        const uint32_t q4 = (uint32_t)(warp & 3);
        const uint32_t lane_addr = tbase + ((q4 * 32u) << 16);
        const uint32_t t = q4 * 32u + (uint32_t)lane;
        const uint32_t krow = tc::smem_u32(sK) + t * kKRow + (uint32_t)(2 * pg) * kKStage;
        auto adv2 = [&](int64_t& sg, int& tix) {   // two tiles on, across segments
            tix += 2;
            while (tix >= nt) {
                tix -= nt;
                ++sg;
            }
        };
        int64_t u_n = (g0 + pg) / nt;              // segment of the next key-row copy
        int ti_n = (int)((g0 + pg) - u_n * nt);
        int64_t pu_n = u_n / P.nrg;                // its pool unit and row group, advanced incrementally
        int rg_n = (int)(u_n - pu_n * P.nrg);
        int kk = 0;
        // copy the key row of this token slot for this group's tile jj into the group's stage kk & 1
        auto issue_k = [&](int jj) {
            if (jj < n) {
                const int64_t tok = (int64_t)ti_n * kTile + t;
                const bool ok = tok < P.n_ctx;
                const int8_t* src = P.p.kq + (pu_n * cap + (ok ? tok : 0)) * kD;
                const uint32_t dst = krow + (uint32_t)(kk & 1) * kKStage;
#pragma unroll
                for (int i = 0; i < 8; ++i) cp_async16(dst + 16u * i, src + 16 * i, ok ? 16u : 0u);
                ti_n += 2;
                while (ti_n >= nt) {
                    ti_n -= nt;
                    if (++rg_n == P.nrg) {
                        rg_n = 0;
                        ++pu_n;
                    }
                }
            }
            ++kk;
            cp_async_commit();
        };
        issue_k(pg);
        int64_t u = (g0 + pg) / nt;                // segment of the current tile
        int ti = (int)((g0 + pg) - u * nt);
        float wscale = pg < n ? unit_wscale(P.p.nmax[u / P.nrg]) : 1.0f;
        const int s = pg;
        int k = 0;
        // The loop always runs to its end so that all 128 threads of the group meet at the same
        // named barriers; after an abort every wait returns at once and the data are ignored.
        for (int j = pg; j < n; j += 2, ++k) {
            const uint32_t ph = (uint32_t)((j >> 1) & 1);
            const int st = j & (kNS - 1);
            const bool valid = (int64_t)ti * kTile + t < P.n_ctx;
            issue_k(j + 2);
            tc::mbar_wait(tc::smem_u32(&M.rfull[st]), (uint32_t)((j / kNS) & 1), abortp, kTimeoutNs);
            const uint8_t* raw = sR + st * kRawStage;
            const uint2 sraw = valid ? *reinterpret_cast<const uint2*>(raw + kRawS + t * 8) : make_uint2(0u, 0u);
            uint32_t w[12];
#pragma unroll
            for (int i = 0; i < 3; ++i) {
                const uint4 x = *reinterpret_cast<const uint4*>(raw + kRawV + t * 48 + 16 * i);
                w[4 * i] = x.x;
                w[4 * i + 1] = x.y;
                w[4 * i + 2] = x.z;
                w[4 * i + 3] = x.w;
            }
            const unsigned short nb = *reinterpret_cast<const unsigned short*>(raw + kRawN + t * 2);
            // the ring stage is refilled by the TMA (async proxy): order these reads before that write
            tc::fence_proxy_async();
            tc::mbar_arrive(tc::smem_u32(&M.rempty[st]));
            cp_async_wait<1>();   // this tile's key row has landed (the next one may be in flight)
            const uint8_t* kr_s = sK + (2 * pg + (k & 1)) * kKStage + t * kKRow;
            // keys: k_hat = s_b * code (times 2^-4 against fp16 overflow) as an exact fp16 pair
            // hi = fp16(k_hat), lo = fp16(k_hat - hi): the product has <= 18 significant bits, hi + lo
            // holds 22, so hi + lo = k_hat and MMA1 over hi then lo gives the exact q . k_hat sums.
            if (j >= 2) tc::mbar_wait(tc::smem_u32(&M.kfree[s]), ph ^ 1u, abortp, kTimeoutNs);
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {   // q8_0 block qq = dims 32qq .. 32qq+31
                const uint32_t sw = (qq < 2 ? sraw.x : sraw.y) >> (16 * (qq & 1));
                __half2 sc = __half2half2(__ushort_as_half((unsigned short)(sw & 0xFFFFu)));
                sc = __hmul2(sc, __half2half2(__ushort_as_half((unsigned short)0x2C00)));  // * 2^-4
                uint32_t rh[16], rl[16];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint4 kr = *reinterpret_cast<const uint4*>(kr_s + 32 * qq + 16 * h);
                    const uint32_t kw[4] = {kr.x, kr.y, kr.z, kr.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        uint32_t c01, c23;
                        i8x4_to_f16x4(kw[e], c01, c23);
                        const __half2 h01 = __hmul2(*reinterpret_cast<const __half2*>(&c01), sc);
                        const __half2 h23 = __hmul2(*reinterpret_cast<const __half2*>(&c23), sc);
                        const __half2 l01 = __hfma2(*reinterpret_cast<const __half2*>(&c01), sc, __hneg2(h01));
                        const __half2 l23 = __hfma2(*reinterpret_cast<const __half2*>(&c23), sc, __hneg2(h23));
                        rh[h * 8 + 2 * e] = *reinterpret_cast<const uint32_t*>(&h01);
                        rh[h * 8 + 2 * e + 1] = *reinterpret_cast<const uint32_t*>(&h23);
                        rl[h * 8 + 2 * e] = *reinterpret_cast<const uint32_t*>(&l01);
                        rl[h * 8 + 2 * e + 1] = *reinterpret_cast<const uint32_t*>(&l23);
                    }
                }
                tc::tmem_st16(lane_addr + kColK + 128u * s + 16u * qq, rh);
                tc::tmem_st16(lane_addr + kColK + 128u * s + 64u + 16u * qq, rl);
            }
            tc::wait_st();
            tc::fence_before();
            tc::mbar_arrive(tc::smem_u32(&M.kfull[s]));
            // values: packed 3-bit codes -> centroids * ||v|| * w in fp16, token-major rows
            const float nw = valid ? __half2float(__ushort_as_half(nb)) * wscale : 0.0f;
            const __half2 nw2 = __float2half2_rn(nw);
            if (j >= 2) tc::mbar_wait(tc::smem_u32(&M.pvfree[s]), ph ^ 1u, abortp, kTimeoutNs);
            const uint32_t vst = tc::smem_u32(sV) + s * 32768;
            store_v_quad<0>(w, lut + lane, vst, t, nw2);
            store_v_quad<4>(w, lut + lane, vst, t, nw2);
            store_v_quad<8>(w, lut + lane, vst, t, nw2);
            store_v_quad<12>(w, lut + lane, vst, t, nw2);
            tc::fence_proxy_async();
            tc::mbar_arrive(tc::smem_u32(&M.vfull[s]));
            const int64_t u_prev = u;
            adv2(u, ti);
            if (u != u_prev && j + 2 < n) wscale = unit_wscale(P.p.nmax[u / P.nrg]);
        }
        cp_async_wait<0>();   // no copy may land in shared memory after the CTA exits
    } else if (warp < 8 + kSmWarps) {
        // =============================== softmax + epilogue (four groups of 16 rows)
        const int grp = (warp - 8) >> 2;        // row group: rows 16*grp .. 16*grp+15
        const int wq = warp & 3;                // TMEM lane quadrant
        const int tt = wq * 32 + lane;          // token slot = TMEM lane (= head-dim index in the epilogue)
        const int si = tid - 256;               // 0 .. kSmThreads-1 over all groups
        const uint32_t lane_addr = tbase + ((uint32_t)(wq * 32) << 16);
        const uint32_t gbar = kBarGroup + grp;
        int R = 0;                               // rows of the current segment
        const int rbase = kGRows * grp;
        int seg = -1;
        int64_t seg_u = -1;
        int64_t u = g0 / nt;
        int ti = (int)(g0 - u * nt) - 1;
        for (int j = 0; j < n; ++j) {
            if (++ti == nt) {
                ti = 0;
                ++u;
            }
            const int s = j & 1;
            const uint32_t ph = (uint32_t)((j >> 1) & 1);
            const bool first = (j == 0) || (ti == 0);
            const bool last = (j == n - 1) || (ti == nt - 1);
            if (first) {
                ++seg;
                seg_u = u;
                const int rg = (int)(u % P.nrg);
                R = min(kNR, P.Rtot - kNR * rg);
                softmax_prologue<QBF16>(P.q, P.p.nmax, u / P.nrg, kNR * rg, P.p.H, P.A, P.Hq, P.G, R, P.scale_log2, sQ,
                                        M, si, warp - 8, lane);
                // the next segment's query rows go to L2 now, so its prologue does not wait on HBM
                const int64_t un = u + 1;
                if (un < (g1 + nt - 1) / nt && si < kNR * 2) {
                    const int rgn = (int)(un % P.nrg);
                    const int rn = kNR * rgn + (si >> 1);          // two threads per row, 128 B each
                    if (rn < P.Rtot && (si >> 1) < kNR) {
                        const int64_t pun = un / P.nrg;
                        const int layer = (int)(pun / P.p.H), kvh = (int)(pun % P.p.H);
                        const uint16_t* qa = P.q + (((int64_t)layer * P.A + rn / P.G) * P.Hq + kvh * P.G + rn % P.G) * kD +
                                             (si & 1) * 64;
                        asm volatile("prefetch.global.L2 [%0];" ::"l"(qa));
                    }
                }
            }
            const float scale_eff = M.scale_eff;
            const bool tail = (int64_t)(ti + 1) * kTile > P.n_ctx;
            const bool valid = (int64_t)ti * kTile + tt < P.n_ctx;
            // -------- logits for this group's 16 rows, d = c * S - m (absolute c * S on a segment's
            // first tile, before the running max exists). S and the per-slot row sums come from TMEM in
            // one round trip and stay in registers; if a new running max is needed (the segment's first
            // tile, or a logit above the max by more than 2^tau) the max is updated and the tile is
            // read again against it, so no tile data is live across the out-of-line update.
            const float2 c2 = make_float2(scale_eff, scale_eff);
            tc::mbar_wait(tc::smem_u32(&M.sfull[s]), ph, abortp, kTimeoutNs);
            tc::fence_after();
            if (j >= 2) tc::mbar_wait(tc::smem_u32(&M.pvfree[s]), ph ^ 1u, abortp, kTimeoutNs);
            uint32_t sd[16], ls[16];   // S, then d, as float bits; per-slot row sums
            bool absolute = first;
            for (;;) {
                tc::tmem_ld16(lane_addr + kColS + 64u * s + rbase, sd);
                if (!first) tc::tmem_ld16(lane_addr + kColL + rbase, ls);
                tc::wait_ld();
                if (first) {   // a segment starts its row sums at zero
#pragma unroll
                    for (int k = 0; k < 16; ++k) ls[k] = 0u;
                }
                const float2* nm2 = reinterpret_cast<const float2*>(&M.nm[rbase]);
                float dmax = -INFINITY;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const float2 sv = make_float2(__uint_as_float(sd[2 * k]), __uint_as_float(sd[2 * k + 1]));
                    float2 d = absolute ? mul2(c2, sv) : fma2(c2, sv, nm2[k]);
                    if (tail && !valid) d = make_float2(-INFINITY, -INFINITY);
                    dmax = fmaxf(dmax, fmaxf(d.x, d.y));
                    sd[2 * k] = __float_as_uint(d.x);
                    sd[2 * k + 1] = __float_as_uint(d.y);
                }
                const bool need = absolute || bar_any(kBarRed + grp, 128, dmax > kTau);
                if (!need) break;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const float v0 = tc::warp_max(__uint_as_float(sd[2 * k]));
                    const float v1 = tc::warp_max(__uint_as_float(sd[2 * k + 1]));
                    if (lane == 2 * k) M.red[grp][wq][2 * k] = v0;
                    if (lane == 2 * k + 1) M.red[grp][wq][2 * k + 1] = v1;
                }
                softmax_new_max(M, grp, tt, rbase, R, gbar, absolute, j, lane_addr, abortp);
                absolute = false;   // the second pass sees every logit at or below the new max
            }
            // -------- probabilities p = 2^d (fp16) and running sums
            const uint32_t prow = tc::smem_u32(sP) + s * 16384;
#pragma unroll
            for (int c8 = 0; c8 < 2; ++c8) {   // 8 rows per 16-byte chunk
                uint32_t pk[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int k = 4 * c8 + e;
                    const float p0 = ex2(__uint_as_float(sd[2 * k])), p1 = ex2(__uint_as_float(sd[2 * k + 1]));
                    const __half2 h = __floats2half2_rn(p0, p1);
                    pk[e] = *reinterpret_cast<const uint32_t*>(&h);
                    const float2 l =
                        add2(make_float2(__uint_as_float(ls[2 * k]), __uint_as_float(ls[2 * k + 1])), make_float2(p0, p1));
                    ls[2 * k] = __float_as_uint(l.x);
                    ls[2 * k + 1] = __float_as_uint(l.y);
                }
                st_shared16(prow + tc::sw128((uint32_t)tt, 16u * (2 * grp + c8)), pk[0], pk[1], pk[2], pk[3]);
            }
            tc::tmem_st16(lane_addr + kColL + rbase, ls);
            tc::fence_before();
            tc::mbar_arrive(tc::smem_u32(&M.sfree[s]));   // S has been read for the last time
            tc::fence_proxy_async();
            tc::mbar_arrive(tc::smem_u32(&M.pfull[s]));

            if (last) {
                // one partial per (segment, CTA): slot = segment + CTA (distinct, at most segments + CTAs)
                softmax_epilogue(M, s, ph, abortp, lane_addr, grp, wq, lane, tt, rbase, R, P.RS, gbar, seg_u + c,
                                 P.ws_acc, P.ws_ml);
            }
        }
    } else if (warp == kWarpMma) {
        // =============================== MMA issuer: an event loop over both chains
        // The whole warp runs the loop with warp-uniform control (barrier tests broadcast from lane
        // 0) and one elected lane issues the MMAs and commits. Issuing from a converged warp instead
        // of a single-lane branch cut the tile period by about a tenth.
        const uint32_t id1 = tc::idesc_f16(128, kNR, false, false);
        const uint32_t id2 = tc::idesc_f16(128, kNR, true, true);
        // Shared-memory descriptors, built once: the start-address field holds address >> 4, so a
        // k-step or stage offset is added to the descriptor itself (every operand is below 256 KB).
        // The issuing warp shares its SM sub-partition with six other warps; every instruction it
        // saves per MMA shortens the tile.
        const bool leader = tc::elect_one();
        uint64_t bq[8];
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) bq[ks] = tc::sdesc(tc::smem_u32(sQ) + (ks / 4) * 8192 + (ks % 4) * 32, 16, 1024);
        const uint64_t av0 = tc::sdesc(tc::smem_u32(sV), 16384, 1024);
        const uint64_t bp0 = tc::sdesc(tc::smem_u32(sP), 16384, 1024);
        const uint32_t tS = tbase + kColS, tK = tbase + kColK, tO = tbase + kColO;
        int j1 = 0, j2 = 0;        // next MMA1 / MMA2 tile
        int seg1 = 0;              // segments whose first MMA1 has been issued
        int ti1 = (int)(g0 % nt), ti2 = ti1;
        bool ok = P.test_stall == 0;
        uint64_t t_last = tc::globaltimer();
        while (ok && j2 < n) {
            bool prog = false;
            if (j1 < n) {
                const int s = j1 & 1;
                const bool f1 = (j1 == 0) || (ti1 == 0);
                const bool r1 = (!f1 || tc::mbar_test(tc::smem_u32(&M.qready), (uint32_t)(seg1 & 1))) &&
                                tc::mbar_test(tc::smem_u32(&M.kfull[s]), (uint32_t)((j1 >> 1) & 1)) &&
                                (j1 < 2 || tc::mbar_test(tc::smem_u32(&M.sfree[s]), (uint32_t)(((j1 - 2) >> 1) & 1)));
                if (__shfl_sync(0xffffffffu, r1 ? 1 : 0, 0)) {
                    tc::fence_after();
                    const uint32_t dS = tS + 64u * s, aK = tK + 128u * s;
                    if (leader) {
                        tc::mma_ts_c<0>(dS, aK, bq[0], id1);   // hi then lo halves of the scaled keys
#pragma unroll
                        for (int ks = 1; ks < 8; ++ks) tc::mma_ts_c<1>(dS, aK + 8u * ks, bq[ks], id1);
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks) tc::mma_ts_c<1>(dS, aK + 64u + 8u * ks, bq[ks], id1);
                        tc::commit(tc::smem_u32(&M.sfull[s]));
                        tc::commit(tc::smem_u32(&M.kfree[s]));
                    }
                    if (f1) ++seg1;
                    if (++ti1 == nt) ti1 = 0;
                    ++j1;
                    prog = true;
                }
            }
            if (j2 < j1) {
                const int s2 = j2 & 1;
                const uint32_t ph2 = (uint32_t)((j2 >> 1) & 1);
                const bool r2 = tc::mbar_test(tc::smem_u32(&M.vfull[s2]), ph2) && tc::mbar_test(tc::smem_u32(&M.pfull[s2]), ph2);
                if (__shfl_sync(0xffffffffu, r2 ? 1 : 0, 0)) {
                    const bool f2 = (j2 == 0) || (ti2 == 0);
                    tc::fence_after();
                    const uint64_t ad = av0 + (uint64_t)(s2 * (32768 >> 4));
                    const uint64_t bd = bp0 + (uint64_t)(s2 * (16384 >> 4));
                    if (leader) {
                        if (f2)
                            tc::mma_ss_c<0>(tO, ad, bd, id2);
                        else
                            tc::mma_ss_c<1>(tO, ad, bd, id2);
#pragma unroll
                        for (int ks = 1; ks < 8; ++ks)
                            tc::mma_ss_c<1>(tO, ad + (uint64_t)(ks * (2048 >> 4)), bd + (uint64_t)(ks * (2048 >> 4)), id2);
                        tc::commit(tc::smem_u32(&M.pvfree[s2]));
                    }
                    if (++ti2 == nt) ti2 = 0;
                    ++j2;
                    prog = true;
                }
            }
            if (prog) {
                t_last = tc::globaltimer();
            } else {
                // lane 0 decides, so the warp leaves the loop together
                const int stop = *abortp ? 1 : (tc::globaltimer() - t_last > kTimeoutNs ? 2 : 0);
                const int stop0 = __shfl_sync(0xffffffffu, stop, 0);
                if (stop0 == 2 && lane == 0) *abortp = 1;
                if (stop0) break;
            }
        }
        if (P.test_stall) *abortp = 0;  // let the other roles discover the stall on their own waits
        if (j1 > 0) {
            // every MMA this warp issued must have completed before the TMEM is freed
            if (leader) tc::commit(tc::smem_u32(&M.done));
            volatile int dummy = 0;
            tc::mbar_wait(tc::smem_u32(&M.done), 0u, &dummy, 50000000ull);
        }
    }

    // ---- tear-down: every role is past its last TMEM access
    tc::fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc::fence_after();
        tc::tmem_dealloc(tbase, kTmemCols);
    }
    if (tid == 0 && M.abort) atomicOr(P.p.status, 1u);
}

int g_num_sms = 0;

int num_sms() {
    if (g_num_sms == 0) {
        int dev = 0, v = 0;
        cudaGetDevice(&dev);
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 1;
        g_num_sms = v;
    }
    return g_num_sms;
}

struct TcPlan {
    int64_t nt, tt, nseg;
    int nctas, nrg, RS;
    size_t slots;   // one partial per (segment, CTA that works on it): slot = segment + CTA
};

TcPlan plan(const PoolView& p, int rows, int64_t n_ctx) {
    TcPlan pl;
    pl.nt = (n_ctx + kTile - 1) / kTile;
    pl.nrg = (rows + kNR - 1) / kNR;
    pl.RS = pl.nrg > 1 ? kNR : rows;
    pl.nseg = (int64_t)p.L * p.H * pl.nrg;
    pl.tt = pl.nseg * pl.nt;
    const int64_t sms = num_sms();
    pl.nctas = (int)(pl.tt < sms ? pl.tt : sms);
    pl.slots = (size_t)(pl.nseg + pl.nctas);
    return pl;
}

}  // namespace

bool attend_tc_supported(const PoolView& p, int rows) { return p.d == kD && rows >= 1; }

size_t attend_tc_workspace(const PoolView& p, int rows, int64_t n_ctx) {
    const TcPlan pl = plan(p, rows, n_ctx);
    return sizeof(float) * pl.slots * (size_t)pl.RS * (size_t)(kD + 2);
}

polykv_status launch_attend_tc(const PoolView& p, polykv_dtype dt, const void* q, float* out, int n_agents,
                               int n_q_heads, int64_t n_ctx, float scale, void* ws, size_t ws_bytes,
                               cudaStream_t stream, const SuffixArgs* sfx) {
    const int G = n_q_heads / p.H;
    const int R = n_agents * G;
    if (!attend_tc_supported(p, R)) return set_error(POLYKV_E_UNSUPPORTED, "tensor-core attend: d=%d rows=%d", p.d, R);
    const TcPlan pl = plan(p, R, n_ctx);
    const size_t need = attend_tc_workspace(p, R, n_ctx);
    if (ws_bytes < need) return set_error(POLYKV_E_BUFFER_TOO_SMALL, "attend: workspace %zu < %zu bytes", ws_bytes, need);
    TcParams P;
    P.p = p;
    P.q = static_cast<const uint16_t*>(q);
    P.ws_acc = static_cast<float*>(ws);
    P.ws_ml = P.ws_acc + pl.slots * (size_t)pl.RS * kD;
    P.n_ctx = n_ctx;
    P.total_tiles = pl.tt;
    P.A = n_agents;
    P.Hq = n_q_heads;
    P.G = G;
    P.Rtot = R;
    P.nrg = pl.nrg;
    P.RS = pl.RS;
    P.nt = (int)pl.nt;
    P.nctas = pl.nctas;
    P.scale_log2 = scale * kLog2eTc;
    // Test hook for the bounded-wait path: POLYKV_TEST_STALL=1 makes every wait on the tensor-core
    // results run out; the CTA then gives up, releases its TMEM and sets the pool's status word.
    const char* stall = getenv("POLYKV_TEST_STALL");
    P.test_stall = (stall && stall[0] == '1') ? 1 : 0;
    auto kern = dt == POLYKV_BF16 ? attend_tc_kernel<true> : attend_tc_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmBytes);
    if (e != cudaSuccess) return set_error(POLYKV_E_CUDA, "attend_tc: smem attribute: %s", cudaGetErrorString(e));
    kern<<<pl.nctas, kThreadsTc, kSmBytes, stream>>>(P);
    e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(POLYKV_E_CUDA, "attend_tc launch: %s", cudaGetErrorString(e));
    if (sfx) {
        const polykv_status ss = launch_attend_suffix(*sfx, dt, p.L, n_agents, p.H, n_q_heads, kD, scale, stream);
        if (ss != POLYKV_OK) return ss;
    }
    MergeLayout ml;
    ml.nrg = pl.nrg;
    ml.RS = pl.RS;
    ml.nt = pl.nt;
    ml.tt = pl.tt;
    ml.nc = pl.nctas;
    return launch_attend_merge(P.ws_acc, P.ws_ml, out, p.L * p.H, p.H, n_agents, n_q_heads, R, 0, ml, kD, stream,
                               sfx ? sfx->acc : nullptr, sfx ? sfx->ml : nullptr);
}

}  // namespace polykv
