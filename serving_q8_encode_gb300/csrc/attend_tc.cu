// Multi-agent decode attention over the shared pool on the 5th-generation
// tensor cores (tcgen05, TMEM accumulators), head_dim 128, any number of
// query rows per kv head (agents x GQA group), taken in row groups of 64.
//
// PolyKV abstract ("PolyKV: A Shared Asymmetrically-Compressed KV Cache Pool
// for Multi-Agent LLM Inference"): N agents read one compressed pool. With 15
// agents x 4 GQA heads = 60 rows per kv head, q.K and p.V are dense
// contractions, so both run as tcgen05.mma with every operand that changes per
// token held in TMEM:
//
//   MMA1, per 128-token tile and q8_0 block b (dims 32b .. 32b+31):
//        S_b^T[token][row] = Kc[token][32 dims] . Q'[row][32 dims]^T
//        with Kc the int8 codes as exact fp16 (A operand in TMEM) and Q' the
//        rows' queries in fp16 scaled by a power of two per row group (bf16
//        queries are then exact); four fp32 accumulators, one per block.
//   softmax (one thread per token and row group; TMEM lane = token):
//        d = sum_b c_b[token] S_b - m with c_b = (block scale) x (logit scale)
//        / (query scale), i.e. the q8_0 scales are applied to the exact
//        per-block dot products; base-2 logits relative to the running max,
//        lazy rescaling only when some d exceeds 2^8 (decided per row group
//        with one OR-reducing barrier); P' = 2^d * ||v|| * w stored as fp16
//        (w a power of two from the pool's per-unit norm maximum, so
//        ||v|| w < 2^7 and P' < 2^15).
//   MMA2: O^T[dim][row] += Cv[dim][token] . P'[token][row]^T, Cv the
//        centroids of the value codes in fp16 (A operand in TMEM, lane =
//        dim), in the ROTATED basis; the merge kernel applies the inverse FWHT
//        once per output row.
//
// The pool's value codes are stored per 32-token group and coordinate (one
// 12-byte string each), so the thread owning TMEM lane j reads the 12 bytes of
// coordinate j for its 32 tokens and writes their centroid pairs straight into
// its lane: neither MMA operand built per tile passes through shared memory.
//
// Data movement: one producer thread streams each tile's key codes (a 2-D
// tensor copy with the 128-byte swizzle, so that every thread's 32-byte key
// block reads conflict-free), value codes, block scales and norms (1-D bulk
// copies) into a 5-stage shared-memory ring. Shared memory also holds the
// queries and P' (the B operands) and a lane-replicated table of centroid
// pairs. Each tile's eight MMA1 and eight MMA2 instructions are issued from one
// asm statement each by an elected lane, with descriptors built once: the
// issuing thread's instruction count, not the tensor core, bounds how fast
// small-N MMAs go.
//
// Work split: one persistent CTA per SM. A segment is one (kv-head unit, row
// group of up to 64 query rows); the (segment, tile) list is cut into one
// contiguous range per CTA, a range that crosses a segment boundary writes one
// softmax partial per segment piece (slot = segment + CTA), and the merge
// kernel combines them. Every pool byte is read from HBM once per row group.
//
// Warp roles (640 threads): warps 0-15 are uniform workers, warp w owning row
// group g = w / 4 (rows 16g .. 16g+15), q8_0 block g, token quarter g and TMEM
// lane quadrant w % 4. Per tile each worker thread converts one 32-code key
// block of its token (lane) into the next tile's key operand, runs the softmax
// of its token for its 16 rows, and converts its coordinate's 32 value codes
// into the value operand. Warp 16 issues the MMAs and owns the TMEM, warp 17
// is the producer and warps 18-19 complete their warpgroup, whose registers go
// to the workers (setmaxnreg). Every mbarrier wait is bounded (2 s); on expiry
// the CTA raises an abort flag, runs its loops to the end with every wait
// returning at once (so named barriers stay matched), waits (bounded) for its
// copies and MMAs, frees its TMEM and sets the pool's status word.
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "polykv_internal.cuh"
#include "tc_ptx.cuh"

namespace polykv {
namespace {

constexpr int kTile = 128;
constexpr int kD = 128;
constexpr int kNR = 64;            // padded rows per segment (MMA N)
constexpr int kGroups = 4;         // row groups = q8_0 blocks = 32-token quarters
constexpr int kGRows = kNR / kGroups;
constexpr int kWorkers = 16;       // worker warps
constexpr int kWarpMma = kWorkers;       // MMA issuer and TMEM owner
constexpr int kWarpTma = kWorkers + 1;   // pool-tile producer
constexpr int kThreadsTc = 32 * (kWorkers + 4);   // + one warpgroup: the MMA warp and three idle warps
constexpr int kRegWorker = 104;    // registers per worker thread after setmaxnreg (launch: 96)
// setmaxnreg draws on the registers the CTA was launched with: 640 x 96 = 61440 >= 512 x 104 + 128 x 56
constexpr int kRegOther = 56;      // the MMA warpgroup's registers after setmaxnreg  // pool tiles prefetched into L2 ahead of MMA1
// named barriers: 1..4 sync one row group, 5..8 OR-reduce within one (never mixed on an id)
constexpr uint32_t kBarGroup = 1, kBarRed = 5;
constexpr float kTau = 8.0f;       // lazy rescale threshold (log2 units): p <= 2^8
constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr float kLog2eTc = 1.4426950408889634f;

// shared memory map (bytes from an 8 KB-aligned base)
constexpr int kStages = 5;                    // pool-tile ring depth
constexpr uint32_t kStKeys = 0;               // stage: key codes [128 tokens][128 B], 128-byte swizzle  16 KB
constexpr uint32_t kStVals = 16384;           //        value codes, 4 groups x 128 dims x 12 B           6 KB
constexpr uint32_t kStScales = 22528;         //        block scales [128 tokens][4] fp16                 1 KB
constexpr uint32_t kStNorms = 23552;          //        norms [128 tokens] fp16                            256 B
constexpr uint32_t kStageTx = 23808;          // bytes the TMA delivers per stage
constexpr uint32_t kStageBytes = 24576;       // stage stride (keys stay 1024-byte aligned)
constexpr uint32_t kSmRing = 0;
constexpr uint32_t kSmQ = kSmRing + kStages * kStageBytes;   // 2 buffers x 2 chunks x [64 rows][128 B]  32 KB
constexpr uint32_t kSmP = kSmQ + 32768;       // 2 buffers x [128 tokens][128 B]                          32 KB
constexpr uint32_t kSmLut = kSmP + 32768;     // 64 code pairs x 32 lanes x 4 B                            8 KB
constexpr uint32_t kSmMisc = kSmLut + 8192;
constexpr uint32_t kMiscBytes = 4096;
constexpr uint32_t kSmBytes = kSmMisc + kMiscBytes + 8192;   // + alignment slack
static_assert(kSmBytes <= 232448, "shared memory budget");
static_assert(kSmLut % 8192 == 0 && kSmQ % 1024 == 0 && kSmP % 1024 == 0 && kStageBytes % 1024 == 0,
              "alignment of the swizzled operands and of the OR-addressed table");
static_assert(kThreadsTc / 32 == kWorkers + 4 && kWorkers % 4 == 0, "workers fill whole warpgroups");
static_assert(kWorkers * 32 * kRegWorker + 128 * kRegOther <= kThreadsTc * 96, "setmaxnreg split");

// TMEM columns
constexpr uint32_t kColS = 0;      // 4 blocks x 64 rows: S_b^T, lane = token
constexpr uint32_t kColK = 256;    // 2 buffers x 64: key codes (fp16 pairs), lane = token
constexpr uint32_t kColV = 384;    // 64: value centroids (fp16 pairs of tokens), lane = dim
constexpr uint32_t kColO = 448;    // 64: O^T, lane = dim
constexpr uint32_t kTmemCols = 512;

struct TcParams {
    CUtensorMap kmap;   // key codes as a 2-D tensor [U * cap rows][128 B], 128-byte swizzle, 128 x 128 boxes
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
    int test_stall;  // test hook: the MMA thread issues nothing, so the workers' waits run out
    float scale_log2;
};

struct Misc {
    float m[kNR];                      // running max per row (log2 units); +inf for padding rows
    float nm[kNR];                     // -m, the addend of the logits (0 before a segment's first tile)
    float delta[kNR];                  // raise of the running max at the last update
    float alpha[kNR];                  // 2^-delta
    float red[kGroups][4][kGRows];     // per (group, lane quadrant, row): partial maxima or row sums
    float qred[kGroups][4];            // per (group, quadrant): query magnitude maxima
    float qc[2][kGroups];              // per query buffer and row group: logit scale / query scale
    int abort;
    int pad;
    uint64_t sfull, kready, pvfull, mma2done, qready[2], done;   // kready: next key operand in TMEM + S read
    uint64_t rfull[kStages], rempty[kStages];
    uint32_t tslot;
};
static_assert(sizeof(Misc) <= kMiscBytes, "misc block");

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
__device__ __forceinline__ float max3f(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// OR of `pred` over the `n` threads of named barrier `id`, which all wait here. Only the vote is
// needed from it (shared-memory hand-offs use their own barriers), so it carries no compiler memory
// clobber and the loads and stores around it may be scheduled across it.
__device__ __forceinline__ bool bar_any(uint32_t id, uint32_t n, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n barrier.cta.red.or.pred q, %2, %3, p;\n"
        " selp.u32 %0, 1, 0, q;\n}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(n));
    return r != 0;
}

// 16-byte shared store as inline asm: it stays ahead of the proxy fence and the mbarrier arrive
// that publish it to the tensor cores.
__device__ __forceinline__ void st_shared16(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
// load from the centroid-pair table, which is read-only after set-up: not volatile, so the compiler
// may schedule it freely
__device__ __forceinline__ uint32_t ld_table32(uint32_t addr) {
    uint32_t v;
    asm("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
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

// One token's q8_0 block (32 int8 codes) -> 16 fp16 pairs in this thread's TMEM lane at `taddr`.
__device__ __forceinline__ void store_key_block(const uint4 (&kc)[2], uint32_t taddr) {
    uint32_t r[16];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const uint32_t w[4] = {kc[h].x, kc[h].y, kc[h].z, kc[h].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) i8x4_to_f16x4(w[e], r[8 * h + 2 * e], r[8 * h + 2 * e + 1]);
    }
    tc::tmem_st16(taddr, r);
}

// Byte offset (times 128) of centroid-pair table entry for tokens (2C, 2C+1): their two 3-bit codes
// are bits 6C .. 6C+5 of the 96-bit string (w2:w1:w0); returns idx << 7 (an entry is 32 lane copies
// of 4 bytes).
template <int C>
__device__ __forceinline__ uint32_t pair_off(uint32_t w0, uint32_t w1, uint32_t w2) {
    constexpr int bit = 6 * C, word = bit >> 5, off = bit & 31;
    const uint32_t lo = word == 0 ? w0 : (word == 1 ? w1 : w2);
    if constexpr (off > 26) {   // the pair straddles two words
        const uint32_t hi = word == 0 ? w1 : w2;
        return __funnelshift_r(lo, hi, off - 7) & 0x1F80u;
    } else if constexpr (off >= 7) {
        return (lo >> (off - 7)) & 0x1F80u;
    } else {
        return (lo << (7 - off)) & 0x1F80u;
    }
}

// The 32 value codes of one coordinate (one 12-byte string) -> 16 fp16 centroid pairs.
__device__ __forceinline__ void value_pairs(uint32_t w0, uint32_t w1, uint32_t w2, uint32_t lut_lane,
                                            uint32_t (&o)[16]) {
#define PKV_PAIR(C) o[C] = ld_table32(lut_lane | pair_off<C>(w0, w1, w2));
    PKV_PAIR(0) PKV_PAIR(1) PKV_PAIR(2) PKV_PAIR(3) PKV_PAIR(4) PKV_PAIR(5) PKV_PAIR(6) PKV_PAIR(7)
    PKV_PAIR(8) PKV_PAIR(9) PKV_PAIR(10) PKV_PAIR(11) PKV_PAIR(12) PKV_PAIR(13) PKV_PAIR(14) PKV_PAIR(15)
#undef PKV_PAIR
}

// MMA1 of one tile, issued by one elected lane of the converged MMA warp: for each q8_0 block b,
// S_b (TMEM columns tS + 64b) = key codes (TMEM columns aK + 16b + 8h, h = 0, 1) . queries (the
// K-major descriptor bq advanced to dims 32b + 16h), then a commit to `bar`. All operand addresses
// are formed inside one asm statement from three values, so issuing costs a few instructions.
__device__ __forceinline__ void issue_mma1(uint32_t tS, uint32_t aK, uint64_t bq, uint32_t idesc, uint32_t bar) {
    asm volatile(
        "{\n .reg .pred P, T, F;\n .reg .b32 d1, d2, d3, a1, a2, a3, a4, a5, a6, a7;\n"
        " .reg .b64 b1, b2, b3, b4, b5, b6, b7;\n"
        " elect.sync _|P, 0xffffffff;\n setp.ne.u32 T, 1, 0;\n setp.ne.u32 F, 0, 0;\n"
        " add.u32 d1, %0, 64;\n add.u32 d2, %0, 128;\n add.u32 d3, %0, 192;\n"
        " add.u32 a1, %1, 8;\n add.u32 a2, %1, 16;\n add.u32 a3, %1, 24;\n add.u32 a4, %1, 32;\n"
        " add.u32 a5, %1, 40;\n add.u32 a6, %1, 48;\n add.u32 a7, %1, 56;\n"
        " add.u64 b1, %2, 2;\n add.u64 b2, %2, 4;\n add.u64 b3, %2, 6;\n add.u64 b4, %2, 512;\n"
        " add.u64 b5, %2, 514;\n add.u64 b6, %2, 516;\n add.u64 b7, %2, 518;\n"
        " @P tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, F;\n"
        " @P tcgen05.mma.cta_group::1.kind::f16 [d1], [a2], b2, %3, F;\n"
        " @P tcgen05.mma.cta_group::1.kind::f16 [d2], [a4], b4, %3, F;\n"
        " @P tcgen05.mma.cta_group::1.kind::f16 [d3], [a6], b6, %3, F;\n"
        " @P tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, T;\n"
        " @P tcgen05.mma.cta_group::1.kind::f16 [d1], [a3], b3, %3, T;\n"
        " @P tcgen05.mma.cta_group::1.kind::f16 [d2], [a5], b5, %3, T;\n"
        " @P tcgen05.mma.cta_group::1.kind::f16 [d3], [a7], b7, %3, T;\n"
        " @P tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%4];\n}" ::"r"(tS),
        "r"(aK), "l"(bq), "r"(idesc), "r"(bar)
        : "memory");
}

// MMA2 of one tile: O (TMEM tO) += value centroids (TMEM columns tV + 8ks) . P' (MN-major descriptor
// bp advanced by 16 tokens = 2 KB per step), ks = 0..7; `fresh` starts the accumulator (a segment's
// first tile); then a commit to `bar`.
__device__ __forceinline__ void issue_mma2(uint32_t tO, uint32_t tV, uint64_t bp, uint32_t idesc, uint32_t fresh,
                                           uint32_t bar) {
    asm volatile(
        "{\n .reg .pred P, T, A0;\n .reg .b32 a1, a2, a3, a4, a5, a6, a7;\n"
        " .reg .b64 b1, b2, b3, b4, b5, b6, b7;\n"
        " elect.sync _|P, 0xffffffff;\n setp.ne.u32 T, 1, 0;\n setp.eq.u32 A0, %4, 0;\n"
        " add.u32 a1, %1, 8;\n add.u32 a2, %1, 16;\n add.u32 a3, %1, 24;\n add.u32 a4, %1, 32;\n"
        " add.u32 a5, %1, 40;\n add.u32 a6, %1, 48;\n add.u32 a7, %1, 56;\n"
        " add.u64 b1, %2, 128;\n add.u64 b2, %2, 256;\n add.u64 b3, %2, 384;\n add.u64 b4, %2, 512;\n"
        " add.u64 b5, %2, 640;\n add.u64 b6, %2, 768;\n add.u64 b7, %2, 896;\n"
        " @P tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, A0;\n"
        " @P tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, T;\n"
        " @P tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], b2, %3, T;\n"
        " @P tcgen05.mma.cta_group::1.kind::f16 [%0], [a3], b3, %3, T;\n"
        " @P tcgen05.mma.cta_group::1.kind::f16 [%0], [a4], b4, %3, T;\n"
        " @P tcgen05.mma.cta_group::1.kind::f16 [%0], [a5], b5, %3, T;\n"
        " @P tcgen05.mma.cta_group::1.kind::f16 [%0], [a6], b6, %3, T;\n"
        " @P tcgen05.mma.cta_group::1.kind::f16 [%0], [a7], b7, %3, T;\n"
        " @P tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%5];\n}" ::"r"(tO),
        "r"(tV), "l"(bp), "r"(idesc), "r"(fresh), "r"(bar)
        : "memory");
}

// One elected lane commits all of this warp's earlier MMAs to `bar`.
__device__ __forceinline__ void commit_elected(uint32_t bar) {
    asm volatile(
        "{\n .reg .pred P;\n elect.sync _|P, 0xffffffff;\n"
        " @P tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}" ::"r"(bar)
        : "memory");
}

// per-unit value scale w = 2^(7 - e), nmax = f * 2^e with f in [0.5, 1): ||v|| * w <= 2^7
__device__ __forceinline__ float unit_wscale(float nmax) {
    int en = 0;
    if (nmax > 0.0f) frexpf(nmax, &en);
    return nmax > 0.0f ? ldexpf(1.0f, 7 - en) : 1.0f;
}

// Position in this CTA's contiguous (segment, tile) list, advanced one tile at a time.
struct Cursor {
    int64_t seg, unit;
    int ti, rg;
    __device__ __forceinline__ void adv(int nt, int nrg) {
        if (++ti == nt) {
            ti = 0;
            ++seg;
            if (++rg == nrg) {
                rg = 0;
                ++unit;
            }
        }
    }
};

// Query rows of one segment handled by this worker thread: row 16g + 4qd + lane/8 of the segment,
// dims 16c .. 16c+15 with c = lane % 8 (two 16-byte loads; zero for padding rows).
__device__ __forceinline__ void q_load(const TcParams& P, const Cursor& c, int g, int qd, int lane, uint4 (&raw)[2]) {
    const int r = kGRows * g + 4 * qd + (lane >> 3), ch = lane & 7;
    const int R0 = c.rg * kNR + r;
    raw[0] = raw[1] = make_uint4(0u, 0u, 0u, 0u);
    if (R0 < P.Rtot) {
        const int layer = (int)(c.unit / P.p.H), kvh = (int)(c.unit % P.p.H);
        const int a = R0 / P.G, gq = R0 % P.G;
        const uint4* src = reinterpret_cast<const uint4*>(
            P.q + (((int64_t)layer * P.A + a) * P.Hq + kvh * P.G + gq) * kD + 16 * ch);
        raw[0] = __ldg(src);
        raw[1] = __ldg(src + 1);
    }
}

// The segment's queries for this row group in fp16, scaled by fq = 2^(15 - e) where the group's
// largest magnitude is f * 2^e (f in [0.5, 1)), into query buffer `qbuf` (the B operand of MMA1,
// K-major, 128-byte swizzle: two chunks of 64 dims x [64 rows][128 B]); the group's combine
// constant (logit scale in log2 units / fq) goes to M.qc. Ends with the buffer published to the
// MMA issuer (one arrival per warp) and a group barrier.
template <bool QBF16>
__device__ __forceinline__ void q_store(const uint4 (&raw)[2], uint32_t qbuf_u, Misc& M, int buf, int g, int qd,
                                        int lane, float scale_log2) {
    float x[16];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const uint32_t w[4] = {raw[h].x, raw[h].y, raw[h].z, raw[h].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if (QBF16) {
                x[8 * h + 2 * e] = __uint_as_float(w[e] << 16);
                x[8 * h + 2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
            } else {
                const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
                x[8 * h + 2 * e] = f.x;
                x[8 * h + 2 * e + 1] = f.y;
            }
        }
    }
    float mx = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) mx = fmaxf(mx, fabsf(x[i]));
    const uint32_t mb = __reduce_max_sync(0xffffffffu, __float_as_uint(mx));   // magnitudes order as uints
    if (lane == 0) M.qred[g][qd] = __uint_as_float(mb);
    tc::named_bar(kBarGroup + g, 128);
    const float qmax = fmaxf(fmaxf(M.qred[g][0], M.qred[g][1]), fmaxf(M.qred[g][2], M.qred[g][3]));
    int eq = 0;
    if (qmax > 0.0f) frexpf(qmax, &eq);
    const float fq = qmax > 0.0f ? ldexpf(1.0f, 15 - eq) : 1.0f;   // qmax * fq in [2^14, 2^15)
    uint32_t hv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const __half2 h2 = __floats2half2_rn(x[2 * i] * fq, x[2 * i + 1] * fq);
        hv[i] = *reinterpret_cast<const uint32_t*>(&h2);
    }
    const int r = kGRows * g + 4 * qd + (lane >> 3), ch = lane & 7;
    const uint32_t rowb = qbuf_u + (uint32_t)(ch >> 2) * 8192u + (uint32_t)r * 128u;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const uint32_t chunk = (uint32_t)(((ch & 3) * 2 + h) ^ (r & 7));
        st_shared16(rowb + (chunk << 4), hv[4 * h], hv[4 * h + 1], hv[4 * h + 2], hv[4 * h + 3]);
    }
    if (qd == 0 && lane == 0) M.qc[buf][g] = scale_log2 / fq;
    tc::fence_proxy_async();
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(tc::smem_u32(&M.qready[buf]));
    tc::named_bar(kBarGroup + g, 128);
}

// Row sums of this row group over the 128 token slots (lanes x quadrants) at the end of a segment
// piece, written with the rows' running maxima as the piece's (m, l) partial; the rows' logit
// addends are reset for the next segment.
__device__ __forceinline__ void write_row_stats(const float2 (&l)[8], Misc& M, int g, int qd, int lane, int R,
                                                float* __restrict__ ml_slot) {
    float v[16];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        v[2 * k] = l[k].x;
        v[2 * k + 1] = l[k].y;
    }
    // transposing butterfly: each round halves the rows a lane keeps and sums them over lane pairs
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const bool up = (lane & 16) != 0;
        const float send = up ? v[k] : v[k + 8], keep = up ? v[k + 8] : v[k];
        v[k] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const bool up = (lane & 8) != 0;
        const float send = up ? v[k] : v[k + 4], keep = up ? v[k + 4] : v[k];
        v[k] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const bool up = (lane & 4) != 0;
        const float send = up ? v[k] : v[k + 2], keep = up ? v[k + 2] : v[k];
        v[k] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    }
    {
        const bool up = (lane & 2) != 0;
        const float send = up ? v[0] : v[1], keep = up ? v[1] : v[0];
        v[0] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
    }
    v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
    const int row = ((lane >> 4) & 1) * 8 + ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 + ((lane >> 1) & 1);
    if ((lane & 1) == 0) M.red[g][qd][row] = v[0];
    // the next segment's first tile takes absolute logits (its addend -m reads 0); every thread of the
    // group has read this tile's addends before the tile's OR barrier
    if (qd == 1 && lane < kGRows) M.nm[kGRows * g + lane] = 0.0f;
    tc::named_bar(kBarGroup + g, 128);
    if (qd == 0 && lane < kGRows) {
        const int r = kGRows * g + lane;
        if (r < R) {
            ml_slot[2 * r] = M.m[r];
            ml_slot[2 * r + 1] = (M.red[g][0][lane] + M.red[g][1][lane]) + (M.red[g][2][lane] + M.red[g][3][lane]);
        }
    }
    // the next segment's first tile rewrites M.red before its own first barrier: no warp of the group may
    // get there while these sums are still being read
    tc::named_bar(kBarGroup + g, 128);
}

template <bool QBF16>
__global__ void __launch_bounds__(kThreadsTc, 1) attend_tc_kernel(const __grid_constant__ TcParams P) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u = tc::smem_u32(smem_raw);
    uint8_t* sm = smem_raw + (((raw_u + 8191u) & ~8191u) - raw_u);
    const uint32_t sm_u = tc::smem_u32(sm);
    uint32_t* lut = reinterpret_cast<uint32_t*>(sm + kSmLut);
    Misc& M = *reinterpret_cast<Misc*>(sm + kSmMisc);
    volatile int* abortp = &M.abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t TT = P.total_tiles;
    const int cta = blockIdx.x;
    const int64_t g0 = (int64_t)cta * TT / P.nctas;
    const int64_t g1 = (int64_t)(cta + 1) * TT / P.nctas;
    const int n = (int)(g1 - g0);
    const int nt = P.nt, nrg = P.nrg;
    Cursor c0;
    c0.seg = g0 / nt;
    c0.ti = (int)(g0 - c0.seg * nt);
    c0.unit = c0.seg / nrg;
    c0.rg = (int)(c0.seg - c0.unit * nrg);

    // ---- set-up: barriers, centroid-pair table, TMEM
    if (tid == 0) {
        tc::mbar_init(tc::smem_u32(&M.sfull), 1);
        tc::mbar_init(tc::smem_u32(&M.kready), kWorkers);
        tc::mbar_init(tc::smem_u32(&M.pvfull), kWorkers);
        tc::mbar_init(tc::smem_u32(&M.mma2done), 1);
        tc::mbar_init(tc::smem_u32(&M.qready[0]), kWorkers);
        tc::mbar_init(tc::smem_u32(&M.qready[1]), kWorkers);
        tc::mbar_init(tc::smem_u32(&M.done), 1);
        for (int st = 0; st < kStages; ++st) {
            tc::mbar_init(tc::smem_u32(&M.rfull[st]), 1);
            tc::mbar_init(tc::smem_u32(&M.rempty[st]), 1);   // released by the MMA warp after pvfull
        }
        M.abort = 0;
        for (int r = 0; r < kNR; ++r) M.nm[r] = 0.0f;   // a segment's first tile takes absolute logits
        tc::mbar_init_fence();
    }
    for (int e = tid; e < 64 * 32; e += kThreadsTc) {
        const int idx = e >> 5;   // two 3-bit codes: the even token in bits 0..2, the odd one in 3..5
        const __half lo = __float2half_rn(centroid_of(idx & 7));
        const __half hi = __float2half_rn(centroid_of(idx >> 3));
        lut[e] = (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
    }
    if (warp == kWarpMma) tc::tmem_alloc(tc::smem_u32(&M.tslot), kTmemCols);
    // the merge kernel (a programmatic dependent) may be scheduled as this grid's CTAs retire; it waits
    // for this grid's completion before it reads the partials
    if (tid == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tbase = M.tslot;

    if (warp < kWorkers) {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegWorker));
        // =============================== workers
        const int g = warp >> 2;                   // row group, key block, token quarter
        const int qd = warp & 3;                   // TMEM lane quadrant
        const int t = qd * 32 + lane;              // TMEM lane: token (keys, softmax) and coordinate (values)
        const uint32_t lane_addr = tbase + ((uint32_t)(qd * 32) << 16);
        const uint32_t lut_lane = sm_u + kSmLut + (uint32_t)lane * 4u;
        const uint32_t rbar = kBarRed + g;
        const uint32_t b_sfull = tc::smem_u32(&M.sfull), b_kready = tc::smem_u32(&M.kready);
        const uint32_t b_m2 = tc::smem_u32(&M.mma2done), b_pv = tc::smem_u32(&M.pvfull);
        // this thread's offsets inside a ring stage
        const uint32_t key_a0 = kStKeys + (uint32_t)t * 128u + ((((uint32_t)(2 * g)) ^ (uint32_t)(t & 7)) << 4);
        const uint32_t key_a1 = kStKeys + (uint32_t)t * 128u + ((((uint32_t)(2 * g + 1)) ^ (uint32_t)(t & 7)) << 4);
        const uint32_t val_off = kStVals + (uint32_t)(g * kD + t) * 12u;
        const uint32_t sc_off = kStScales + (uint32_t)t * 8u;
        const uint32_t nv_off = kStNorms + (uint32_t)t * 2u;
        // the last tile of a segment holds tokens [(nt - 1) * 128, n_ctx): this thread's token is valid there
        // only if t < tail_lim
        const int tail_lim = (int)(P.n_ctx - (int64_t)(nt - 1) * kTile);
        auto seg_cursor = [&](int64_t seg, Cursor& c) {
            c.seg = seg;
            c.unit = seg / nrg;
            c.rg = (int)(seg - c.unit * nrg);
            c.ti = 0;
        };

        // prologue: the first segments' queries, then tile 0's key operand (-> kready phase 0)
        int ti_c = c0.ti;                                   // tile index inside its segment: tiles i, i+1, i+2
        int ti_1 = ti_c + 1 == nt ? 0 : ti_c + 1;
        int ti_2 = ti_1 + 1 == nt ? 0 : ti_1 + 1;
        int k_c = 0;                                        // segment ordinals (from this CTA's first) of i, i+1, i+2
        int k_1 = ti_1 == 0 ? 1 : 0;
        int k_2 = k_1 + (ti_2 == 0 ? 1 : 0);
        {
            uint4 qr[2];
            q_load(P, c0, g, qd, lane, qr);
            q_store<QBF16>(qr, sm_u + kSmQ, M, 0, g, qd, lane, P.scale_log2);
            if (n > 1 && ti_1 == 0) {
                Cursor c1;
                seg_cursor(c0.seg + 1, c1);
                q_load(P, c1, g, qd, lane, qr);
                q_store<QBF16>(qr, sm_u + kSmQ + 16384u, M, 1, g, qd, lane, P.scale_log2);
            }
            tc::mbar_wait(tc::smem_u32(&M.rfull[0]), 0u, abortp, kTimeoutNs);
            uint4 kc[2];
            kc[0] = *reinterpret_cast<const uint4*>(sm + kSmRing + key_a0);
            kc[1] = *reinterpret_cast<const uint4*>(sm + kSmRing + key_a1);
            store_key_block(kc, lane_addr + kColK + 16u * g);
            tc::wait_st();
            tc::fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(b_kready);
        }

        int st_c = 0, st_1 = kStages > 1 ? 1 : 0;          // ring stages of tiles i and i+1
        uint32_t ph_1 = 0;                                  // phase of tile i+1's stage
        float2 l[8];
        float cst = 0.0f, wsc = 1.0f;
        int R = 0;
        int64_t slot_c = 0;
        // a finished segment piece whose O is read out at the next tile (after its last MMA2)
        bool epi = false;
        int epi_R = 0;
        float epi_inv_w = 1.0f;
        int64_t epi_slot = 0;
        for (int i = 0; i < n; ++i) {
            const bool first = (i == 0) || (ti_c == 0);
            const bool last = (i == n - 1) || (ti_c == nt - 1);
            if (first) {
                Cursor cs;
                seg_cursor(c0.seg + k_c, cs);
                R = min(kNR, P.Rtot - kNR * cs.rg);
                cst = M.qc[k_c & 1][g];
                wsc = unit_wscale(P.p.nmax[cs.unit]);
                slot_c = cs.seg + cta;   // one partial per (segment, CTA): distinct
#pragma unroll
                for (int k = 0; k < 8; ++k) l[k] = make_float2(0.0f, 0.0f);
            }
            const uint8_t* stgp = sm + kSmRing + (uint32_t)st_c * kStageBytes;
            const uint8_t* stgp1 = sm + kSmRing + (uint32_t)st_1 * kStageBytes;
            // queries of tile i+2's segment, if it starts one (loaded now, stored at the end)
            const bool qprep = (i + 2 < n) && ti_2 == 0;
            uint4 qr[2];
            if (qprep) {
                Cursor cq;
                seg_cursor(c0.seg + k_2, cq);
                q_load(P, cq, g, qd, lane, qr);
            }

            // -- b. S(i) = MMA1(i); tile i+1's pool data (keys)
            tc::mbar_wait(b_sfull, (uint32_t)(i & 1), abortp, kTimeoutNs);
            tc::fence_after();
            const bool more = i + 1 < n;
            if (more) tc::mbar_wait(tc::smem_u32(&M.rfull[st_1]), ph_1, abortp, kTimeoutNs);

            // -- c. logits d = sum_b c_b S_b - m (absolute on a segment's first tile: m = 0 then), with
            //       tile i+1's key operand converted while the S loads are in flight
            const uint2 scw = *reinterpret_cast<const uint2*>(stgp + sc_off);
            uint4 kc[2];
            kc[0] = *reinterpret_cast<const uint4*>(stgp1 + key_a0);
            kc[1] = *reinterpret_cast<const uint4*>(stgp1 + key_a1);
            float2 d[8];
            {
                const float4* nmv = reinterpret_cast<const float4*>(&M.nm[kGRows * g]);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float4 v = nmv[k];
                    d[2 * k] = make_float2(v.x, v.y);
                    d[2 * k + 1] = make_float2(v.z, v.w);
                }
                uint32_t sa[16], sb[16];
                tc::tmem_ld16(lane_addr + kColS + 16u * g, sa);
                tc::tmem_ld16(lane_addr + kColS + 64u + 16u * g, sb);
                const float2 s01 = __half22float2(*reinterpret_cast<const __half2*>(&scw.x));
                const float2 s23 = __half22float2(*reinterpret_cast<const __half2*>(&scw.y));
                const float cb0 = s01.x * cst, cb1 = s01.y * cst, cb2 = s23.x * cst, cb3 = s23.y * cst;
                tc::wait_ld();
                const float2 c0x = make_float2(cb0, cb0), c1x = make_float2(cb1, cb1);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    d[k] = fma2(c0x, make_float2(__uint_as_float(sa[2 * k]), __uint_as_float(sa[2 * k + 1])), d[k]);
                    d[k] = fma2(c1x, make_float2(__uint_as_float(sb[2 * k]), __uint_as_float(sb[2 * k + 1])), d[k]);
                }
                tc::tmem_ld16(lane_addr + kColS + 128u + 16u * g, sa);
                tc::tmem_ld16(lane_addr + kColS + 192u + 16u * g, sb);
                // tile i+1's key operand into the buffer MMA1(i-1) has finished reading
                if (more) store_key_block(kc, lane_addr + kColK + (uint32_t)((i + 1) & 1) * 64u + 16u * g);
                tc::wait_ld();
                tc::wait_st();
                // S(i) has been read for the last time and the next key operand is in place: MMA1(i+1)
                tc::fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(b_kready);
                const float2 c2x = make_float2(cb2, cb2), c3x = make_float2(cb3, cb3);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    d[k] = fma2(c2x, make_float2(__uint_as_float(sa[2 * k]), __uint_as_float(sa[2 * k + 1])), d[k]);
                    d[k] = fma2(c3x, make_float2(__uint_as_float(sb[2 * k]), __uint_as_float(sb[2 * k + 1])), d[k]);
                }
            }
            const bool valid = ti_c != nt - 1 || t < tail_lim;
            if (!valid) {
#pragma unroll
                for (int k = 0; k < 8; ++k) d[k] = make_float2(-INFINITY, -INFINITY);
            }
            float dmax = -INFINITY;
#pragma unroll
            for (int k = 0; k < 8; ++k) dmax = max3f(dmax, d[k].x, d[k].y);
            // -- lazy rescale: only when some logit of the row group exceeds its running max by 2^tau
            bool resc = false;
            if (first || bar_any(rbar, 128, dmax > kTau)) {
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const float v0 = tc::warp_max(d[k].x);
                    const float v1 = tc::warp_max(d[k].y);
                    if (lane == 2 * k) M.red[g][qd][2 * k] = v0;
                    if (lane == 2 * k + 1) M.red[g][qd][2 * k + 1] = v1;
                }
                tc::named_bar(kBarGroup + g, 128);
                if (qd == 0 && lane < kGRows) {
                    const int r = kGRows * g + lane;
                    const float mt = fmaxf(fmaxf(M.red[g][0][lane], M.red[g][1][lane]),
                                           fmaxf(M.red[g][2][lane], M.red[g][3][lane]));
                    float dl = 0.0f, al = 1.0f;
                    if (first) {
                        dl = r < R ? mt : INFINITY;   // padding rows: d = -inf from now on
                        M.m[r] = dl;
                        M.nm[r] = -dl;
                    } else if (r < R && mt > 0.0f) {
                        dl = mt;
                        al = ex2(-mt);
                        M.m[r] += mt;
                        M.nm[r] = -M.m[r];
                    }
                    M.delta[r] = dl;
                    M.alpha[r] = al;
                }
                tc::named_bar(kBarGroup + g, 128);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const float2 dl = *reinterpret_cast<const float2*>(&M.delta[kGRows * g + 2 * k]);
                    d[k] = make_float2(d[k].x - dl.x, d[k].y - dl.y);
                    if (!first) l[k] = mul2(l[k], *reinterpret_cast<const float2*>(&M.alpha[kGRows * g + 2 * k]));
                }
                resc = !first;
            }
            // -- d. probabilities: p = 2^d summed into l; P' = p * ||v|| * w in fp16
            const uint32_t nvb = *reinterpret_cast<const unsigned short*>(stgp + nv_off);
            const uint32_t* vsrc = reinterpret_cast<const uint32_t*>(stgp + val_off);
            const uint32_t w0 = vsrc[0], w1 = vsrc[1], w2 = vsrc[2];
            const float nwf = valid ? __half2float(__ushort_as_half((unsigned short)nvb)) * wsc : 0.0f;
            const float2 nw2 = make_float2(nwf, nwf);
            uint32_t pk[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float2 pr = make_float2(ex2(d[k].x), ex2(d[k].y));
                l[k] = add2(l[k], pr);
                const float2 pw = mul2(pr, nw2);
                const __half2 h = __floats2half2_rn(pw.x, pw.y);
                pk[k] = *reinterpret_cast<const uint32_t*>(&h);
            }
            // -- e. value operand of tile i: this coordinate's centroids for token quarter g
            uint32_t vv[16];
            value_pairs(w0, w1, w2, lut_lane, vv);

            {
                // P'(i) into buffer i & 1, last read by MMA2(i-2), which this thread saw complete in the
                // previous iteration. P'^T rows (token t) of the MN-major B operand, 128-byte swizzle:
                // this thread's 16 rows are the 16-byte chunks 2g and 2g+1 of the token's 128-byte row
                const uint32_t prow = sm_u + kSmP + (uint32_t)(i & 1) * 16384u + (uint32_t)t * 128u;
                st_shared16(prow + ((uint32_t)((2 * g) ^ (t & 7)) << 4), pk[0], pk[1], pk[2], pk[3]);
                st_shared16(prow + ((uint32_t)((2 * g + 1) ^ (t & 7)) << 4), pk[4], pk[5], pk[6], pk[7]);
            }
            // -- f. after MMA2(i-1): write out a finished piece's O, rescale O, publish V'(i)
            if (i > 0) {
                tc::mbar_wait(b_m2, (uint32_t)((i - 1) & 1), abortp, kTimeoutNs);
                tc::fence_after();
            }
            if (epi) {
                uint32_t ov[16];
                tc::tmem_ld16(lane_addr + kColO + 16u * g, ov);
                tc::wait_ld();
                float* acc = P.ws_acc + epi_slot * P.RS * kD;
#pragma unroll
                for (int k = 0; k < kGRows; ++k) {
                    const int r = kGRows * g + k;
                    if (r < epi_R) acc[r * kD + t] = __uint_as_float(ov[k]) * epi_inv_w;
                }
                epi = false;
            }
            if (resc) {
                uint32_t ox[16];
                tc::tmem_ld16(lane_addr + kColO + 16u * g, ox);
                tc::wait_ld();
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    ox[k] = __float_as_uint(__uint_as_float(ox[k]) * M.alpha[kGRows * g + k]);
                tc::tmem_st16(lane_addr + kColO + 16u * g, ox);
            }
            tc::tmem_st16(lane_addr + kColV + 16u * g, vv);
            tc::wait_st();
            tc::fence_before();
            // orders this thread's reads of ring stage i (and P' writes) before the async proxy: the MMA
            // warp releases the stage to the TMA once every worker has arrived here
            tc::fence_proxy_async();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(b_pv);
            // -- g. end of a segment piece: its (m, l) now, its O after MMA2(i) (next tile or below)
            if (last) {
                write_row_stats(l, M, g, qd, lane, R, P.ws_ml + slot_c * P.RS * 2);
                epi = true;
                epi_R = R;
                epi_inv_w = 1.0f / wsc;
                epi_slot = slot_c;
            }
            // -- h. queries of tile i+2's segment (its buffer was last used by the segment before
            //       tile i+1's, whose MMA1s have all completed)
            if (qprep)
                q_store<QBF16>(qr, sm_u + kSmQ + (uint32_t)(k_2 & 1) * 16384u, M, k_2 & 1, g, qd, lane, P.scale_log2);
            // advance the per-tile counters
            st_c = st_1;
            if (++st_1 == kStages) {
                st_1 = 0;
                ph_1 ^= 1u;
            }
            ti_c = ti_1;
            ti_1 = ti_2;
            k_c = k_1;
            k_1 = k_2;
            if (++ti_2 == nt) {
                ti_2 = 0;
                ++k_2;
            }
        }
        if (epi) {
            tc::mbar_wait(b_m2, (uint32_t)((n - 1) & 1), abortp, kTimeoutNs);
            tc::fence_after();
            uint32_t ov[16];
            tc::tmem_ld16(lane_addr + kColO + 16u * g, ov);
            tc::wait_ld();
            float* acc = P.ws_acc + epi_slot * P.RS * kD;
#pragma unroll
            for (int k = 0; k < kGRows; ++k) {
                const int r = kGRows * g + k;
                if (r < epi_R) acc[r * kD + t] = __uint_as_float(ov[k]) * epi_inv_w;
            }
        }
        tc::fence_before();
    } else {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegOther));
        if (warp == kWarpMma) {
            // =========================== MMA issuer: the warp runs the loop converged; one elected
            // lane issues each tile's eight MMAs and its commit from a single asm statement
            const uint32_t id1 = tc::idesc_f16(128, kNR, false, false);   // A (keys) in TMEM, B (queries) K-major
            const uint32_t id2 = tc::idesc_f16(128, kNR, false, true);    // A (values) in TMEM, B (P') MN-major
            const uint64_t bq0 = tc::sdesc(sm_u + kSmQ, 16, 1024);
            const uint64_t bp0 = tc::sdesc(sm_u + kSmP, 16384, 1024);
            const uint32_t tS = tbase + kColS, tK = tbase + kColK, tV = tbase + kColV, tO = tbase + kColO;
            const uint32_t b_sfull = tc::smem_u32(&M.sfull), b_m2 = tc::smem_u32(&M.mma2done);
            // bounded wait by lane 0, result broadcast so that the warp stays converged; the issuer polls
            // (test_wait) instead of suspending, because its wake-up latency sits on the per-tile chain
            auto wait0 = [&](uint64_t& bar, uint32_t ph) -> bool {
                int ok = 1;
                if (lane == 0) ok = tc::mbar_poll(tc::smem_u32(&bar), ph, abortp, kTimeoutNs) ? 1 : 0;
                return __shfl_sync(0xffffffffu, ok, 0) != 0;
            };
            int ti = c0.ti;
            int k = 0;                 // segment ordinal of tile i
            int st_prev = 0;           // ring stage of tile i-1
            bool prev_first = true;
            int issued = 0;
            bool ok = P.test_stall == 0;
            for (int i = 0; i <= n && ok; ++i) {
                bool cur_first = false;
                if (i < n) {
                    cur_first = (i == 0) || (ti == 0);
                    if (cur_first && i > 0) ++k;
                    // tile i's key operand is in TMEM and S(i-1) has been read
                    ok = wait0(M.kready, (uint32_t)(i & 1));
                    if (ok && cur_first) ok = wait0(M.qready[k & 1], (uint32_t)((k >> 1) & 1));
                    if (!ok) break;
                    tc::fence_after();
                    issue_mma1(tS, tK + (uint32_t)(i & 1) * 64u, bq0 + (uint64_t)((k & 1) * (16384 >> 4)), id1, b_sfull);
                    issued = 1;
                }
                if (i > 0) {
                    ok = wait0(M.pvfull, (uint32_t)((i - 1) & 1));
                    if (!ok) break;
                    tc::fence_after();
                    // every worker has read ring stage i-1 for the last time: the TMA may refill it
                    if (lane == 0) tc::mbar_arrive(tc::smem_u32(&M.rempty[st_prev]));
                    issue_mma2(tO, tV, bp0 + (uint64_t)(((i - 1) & 1) * (16384 >> 4)), id2, prev_first ? 1u : 0u, b_m2);
                }
                __syncwarp();
                prev_first = cur_first;
                if (i < n) {
                    if (++ti == nt) ti = 0;
                    st_prev = i % kStages;
                }
            }
            if (P.test_stall) *abortp = 0;   // let the workers discover the stall on their own waits
            if (issued) {
                // every MMA this warp issued must have completed before the TMEM is freed
                commit_elected(tc::smem_u32(&M.done));
                int fin = 1;
                if (lane == 0) {
                    volatile int dummy = 0;
                    fin = tc::mbar_wait(tc::smem_u32(&M.done), 0u, &dummy, 50000000ull) ? 1 : 0;
                    if (!fin) *abortp = 1;   // reported through the pool's status word
                }
                __syncwarp();
            }
        } else if (warp == kWarpTma && lane == 0) {
            // =========================== producer: each tile's key codes (2-D tensor copy, 128-byte
            // swizzle), value codes, scales and norms (1-D bulk copies) into the ring
            Cursor c = c0;
            int issued = 0;
            for (int j = 0; j < n && !*abortp; ++j) {
                const int st = j % kStages;
                if (j >= kStages &&
                    !tc::mbar_wait(tc::smem_u32(&M.rempty[st]), (uint32_t)(((j / kStages) - 1) & 1), abortp, kTimeoutNs))
                    break;
                const int64_t row = c.unit * P.p.cap + (int64_t)c.ti * kTile;   // pool row of token 0
                const uint32_t dst = sm_u + kSmRing + (uint32_t)st * kStageBytes;
                const uint32_t bar = tc::smem_u32(&M.rfull[st]);
                tc::mbar_arrive_expect_tx(bar, kStageTx);
                tc::tma_2d_g2s(dst + kStKeys, &P.kmap, 0, (int32_t)row, bar);
                tc::bulk_g2s(dst + kStVals, P.p.vc + row * (3 * kD / 8), kTile * 3 * kD / 8, bar);
                tc::bulk_g2s(dst + kStScales, P.p.ks + row * (kD / kQ8Block), kTile * (kD / kQ8Block) * 2, bar);
                tc::bulk_g2s(dst + kStNorms, P.p.vn + row, kTile * 2, bar);
                issued = j + 1;
                c.adv(nt, nrg);
            }
            // drain: no copy may land in shared memory after the CTA has exited
            for (int j = issued > kStages ? issued - kStages : 0; j < issued; ++j) {
                volatile int dummy = 0;
                tc::mbar_wait(tc::smem_u32(&M.rfull[j % kStages]), (uint32_t)((j / kStages) & 1), &dummy, 50000000ull);
            }
        }
    }

    // ---- tear-down: every role is past its last TMEM access
    __syncthreads();
    if (warp == kWarpMma) {
        tc::fence_after();
        tc::tmem_dealloc(tbase, kTmemCols);
    }
    if (tid == 0 && M.abort) atomicOr(P.p.status, 1u);
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
    const int64_t sms = device_sm_count();
    pl.nctas = (int)(pl.tt < sms ? pl.tt : sms);
    pl.slots = (size_t)(pl.nseg + pl.nctas);
    return pl;
}

// cuTensorMapEncodeTiled from the driver, looked up once (no link-time dependency on libcuda)
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// The pool's key codes as a 2-D uint8 tensor [U * cap rows][128 B] read in 128 x 128 boxes with the
// 128-byte swizzle (16-byte chunk c of row r lands at chunk c ^ (r % 8)).
polykv_status key_tensor_map(const PoolView& p, CUtensorMap* m) {
    const int64_t rows = (int64_t)p.L * p.H * p.cap;
    if (rows >= ((int64_t)1 << 31)) return set_error(POLYKV_E_UNSUPPORTED, "attend_tc: pool too large (%lld rows)", (long long)rows);
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return set_error(POLYKV_E_CUDA, "attend_tc: cuTensorMapEncodeTiled is not available");
    const cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)kD};
    const cuuint32_t box[2] = {(cuuint32_t)kD, (cuuint32_t)kTile};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, (void*)p.kq, dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return set_error(POLYKV_E_CUDA, "attend_tc: tensor map encode failed (%d)", (int)r);
    return POLYKV_OK;
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
    if (pl.nt > 0x7FFFFFFF) return set_error(POLYKV_E_UNSUPPORTED, "attend: context too long");
    TcParams P;
    const polykv_status ms = key_tensor_map(p, &P.kmap);
    if (ms != POLYKV_OK) return ms;
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
