// Private per-agent keys/values attended together with the shared compressed pool under ONE
// softmax: a suffix of uncompressed recent tokens, or (query-chunk mode) a chunk of query tokens
// that each carry their own key/value, seen causally.
//
// Each agent appends its own recent tokens after the shared context; those
// are not part of the compressed pool (the PolyKV abstract's pool is the shared
// context written once). For every (layer, agent, kv head) the kernels here
// score the agent's query heads against its own keys and accumulate its values
// in the ORIGINAL basis, producing one online-softmax partial (running max m in
// log2 units, sum l, unnormalised accumulator) per query row. The merge kernel
// combines it with the pool partials (whose accumulators are in the rotated
// basis) after the pool part's inverse FWHT.
//
// suffix_mma and chunk_mma (up to 8 query heads per kv head) run on warp-level
// tensor-core MMAs with register-direct loads; suffix_partial and chunk_partial
// (CUDA cores, fp32) take more query heads per kv head.
#include <cmath>

#include "polykv_internal.cuh"

namespace polykv {
namespace {

constexpr int kSfxTile = 128;   // suffix tokens per tile (one per thread for the scores)
constexpr int kSfxThreads = 128;

__device__ __forceinline__ float bits_to_float(uint16_t b, bool bf16) {
    return bf16 ? __uint_as_float((uint32_t)b << 16) : __half2float(__ushort_as_half(b));
}

// Shared-memory tile of the suffix: keys with rows padded by 16 bytes (a thread reads its token's row;
// the padding spreads eight consecutive rows over distinct banks) and values unpadded (a thread reads
// one column; consecutive threads read consecutive 2-byte elements).
template <int D>
struct SfxTileSmem {
    static constexpr int kKRow = 2 * D + 16;
    static constexpr int kKBytes = kSfxTile * kKRow;
    static constexpr int kVBytes = kSfxTile * 2 * D;
    static constexpr int kBytes = kKBytes + kVBytes;
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// grid: one block per (layer, agent, kv head); block: 128 threads. Each 128-token tile of the agent's
// keys and values is copied into shared memory with coalesced 16-byte asynchronous copies; the scores
// (thread = token) and the value accumulation (thread = head dim) then read shared memory only.
template <int D, int GMAX, bool BF16>
__global__ void __launch_bounds__(kSfxThreads) suffix_partial(const uint16_t* __restrict__ q,
                                                              const uint16_t* __restrict__ sk,
                                                              const uint16_t* __restrict__ sv, int A, int H, int Hq,
                                                              int64_t S, float scale_log2, float* __restrict__ acc_out,
                                                              float* __restrict__ ml_out) {
    using T = SfxTileSmem<D>;
    extern __shared__ __align__(16) unsigned char sfx_smem[];
    __shared__ __align__(16) float qs[GMAX][D];
    __shared__ __align__(16) float ps[kSfxTile][GMAX];   // probabilities, token-major
    __shared__ float red[4][GMAX];
    __shared__ float m_s[GMAX], l_s[GMAX], al_s[GMAX];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = Hq / H;
    const int unit = blockIdx.x;                    // (layer * A + a) * H + h
    const int h = unit % H;
    const int la = unit / H;                        // layer * A + a
    const uint16_t* kbase = sk + (int64_t)unit * S * D;
    const uint16_t* vbase = sv + (int64_t)unit * S * D;
    const uint32_t ks_u = (uint32_t)__cvta_generic_to_shared(sfx_smem);
    const uint32_t vs_u = ks_u + T::kKBytes;
    const uint16_t* Vs = reinterpret_cast<const uint16_t*>(sfx_smem + T::kKBytes);

    for (int i = tid; i < GMAX * D; i += kSfxThreads) {
        const int g = i / D, j = i % D;
        qs[g][j] = g < G ? bits_to_float(q[((int64_t)la * Hq + h * G + g) * D + j], BF16) : 0.0f;
    }
    if (tid < GMAX) {
        m_s[tid] = -INFINITY;
        l_s[tid] = 0.0f;
    }
    constexpr int CPT = (D + kSfxThreads - 1) / kSfxThreads;   // accumulator columns per thread
    float acc[GMAX][CPT];
#pragma unroll
    for (int g = 0; g < GMAX; ++g)
#pragma unroll
        for (int c = 0; c < CPT; ++c) acc[g][c] = 0.0f;

    constexpr int kChunksPerRow = D / 8;            // 16-byte chunks per key or value row
    for (int64_t t0 = 0; t0 < S; t0 += kSfxTile) {
        const int tmax = (int)((S - t0) < kSfxTile ? (S - t0) : kSfxTile);
        // ---- the tile's keys and values into shared memory (rows past the suffix are not copied)
        for (int c = tid; c < tmax * kChunksPerRow; c += kSfxThreads) {
            const int row = c / kChunksPerRow, col = c - row * kChunksPerRow;
            const int64_t goff = (t0 + row) * D + col * 8;
            cp_async16(ks_u + (uint32_t)(row * T::kKRow + col * 16), kbase + goff);
            cp_async16(vs_u + (uint32_t)(row * 2 * D + col * 16), vbase + goff);
        }
        cp_async_wait_all();
        __syncthreads();

        // ---- scores: thread = token
        const bool valid = tid < tmax;
        float x[GMAX];
#pragma unroll
        for (int g = 0; g < GMAX; ++g) x[g] = 0.0f;
        if (valid) {
            const unsigned char* krow = sfx_smem + tid * T::kKRow;
#pragma unroll 4
            for (int c = 0; c < kChunksPerRow; ++c) {
                const uint4 w = *reinterpret_cast<const uint4*>(krow + 16 * c);
                const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
                float kf[8];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    kf[2 * e] = bits_to_float((uint16_t)(wv[e] & 0xFFFFu), BF16);
                    kf[2 * e + 1] = bits_to_float((uint16_t)(wv[e] >> 16), BF16);
                }
#pragma unroll
                for (int g = 0; g < GMAX; ++g) {
                    const float4 qa = *reinterpret_cast<const float4*>(&qs[g][8 * c]);
                    const float4 qb = *reinterpret_cast<const float4*>(&qs[g][8 * c + 4]);
                    float s = x[g];
                    s = fmaf(qa.x, kf[0], s);
                    s = fmaf(qa.y, kf[1], s);
                    s = fmaf(qa.z, kf[2], s);
                    s = fmaf(qa.w, kf[3], s);
                    s = fmaf(qb.x, kf[4], s);
                    s = fmaf(qb.y, kf[5], s);
                    s = fmaf(qb.z, kf[6], s);
                    s = fmaf(qb.w, kf[7], s);
                    x[g] = s;
                }
            }
        }
#pragma unroll
        for (int g = 0; g < GMAX; ++g) {
            x[g] = valid ? x[g] * scale_log2 : -INFINITY;
            float v = x[g];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
            if (lane == 0) red[warp][g] = v;
        }
        __syncthreads();
        if (tid < GMAX) {
            const float mt = fmaxf(fmaxf(red[0][tid], red[1][tid]), fmaxf(red[2][tid], red[3][tid]));
            const float mo = m_s[tid];
            const float mn = fmaxf(mo, mt);
            al_s[tid] = mo == -INFINITY ? 0.0f : exp2f(mo - mn);
            m_s[tid] = mn;
        }
        __syncthreads();
#pragma unroll
        for (int g = 0; g < GMAX; ++g) {
            const float p = valid ? exp2f(x[g] - m_s[g]) : 0.0f;
            ps[tid][g] = p;
            float v = p;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            if (lane == 0) red[warp][g] = v;
        }
        __syncthreads();
        if (tid < GMAX) l_s[tid] = l_s[tid] * al_s[tid] + red[0][tid] + red[1][tid] + red[2][tid] + red[3][tid];
        // ---- values: thread = column
#pragma unroll
        for (int c = 0; c < CPT; ++c) {
            const int j = tid + c * kSfxThreads;
            if (j < D) {
#pragma unroll
                for (int g = 0; g < GMAX; ++g) acc[g][c] *= al_s[g];
#pragma unroll 4
                for (int tt = 0; tt < tmax; ++tt) {
                    const float vv = bits_to_float(Vs[tt * D + j], BF16);
#pragma unroll
                    for (int g4 = 0; g4 < GMAX; g4 += 4) {
                        const float4 p4 = *reinterpret_cast<const float4*>(&ps[tt][g4]);
                        acc[g4][c] = fmaf(p4.x, vv, acc[g4][c]);
                        acc[g4 + 1][c] = fmaf(p4.y, vv, acc[g4 + 1][c]);
                        acc[g4 + 2][c] = fmaf(p4.z, vv, acc[g4 + 2][c]);
                        acc[g4 + 3][c] = fmaf(p4.w, vv, acc[g4 + 3][c]);
                    }
                }
            }
        }
        __syncthreads();   // the tile's shared memory is reused by the next tile's copies
    }
    // partial per query head hq = h*G + g of agent a
#pragma unroll
    for (int c = 0; c < CPT; ++c) {
        const int j = tid + c * kSfxThreads;
        if (j < D)
            for (int g = 0; g < G && g < GMAX; ++g) acc_out[((int64_t)la * Hq + h * G + g) * D + j] = acc[g][c];
    }
    if (tid < G) {
        ml_out[((int64_t)la * Hq + h * G + tid) * 2] = m_s[tid];
        ml_out[((int64_t)la * Hq + h * G + tid) * 2 + 1] = l_s[tid];
    }
}

// ---------------------------------------------------------------- suffix on warp-level MMAs (G <= 8)
// The suffix is plain bf16 or f16 K/V, so it is read at HBM rate only if every byte goes straight from a
// wide load into arithmetic. One CTA of four warps takes one (layer, agent, kv head) unit at a time
// (persistent over units); warp w takes the w-th quarter of the unit's 16-token steps and keeps its
// online-softmax state in registers; the four warp partials are combined in shared memory.
//
// Per 16-token step, with m16n8k16 MMAs in the inputs' own type (products exact, fp32 sums):
//   scores  S[row][token] = Q[row][dims] . K[token][dims]^T: M = the unit's G query rows (zero-padded
//           to 16), N = 8 tokens, K = 16 dims per step. The head dimension is permuted identically for
//           Q and K (the dot product does not change): at k-step s, lane quad position t owns the four
//           dims D/4 * t + 4s + {0..3}, so each lane reads one contiguous quarter of a key row.
//   values  O^T[dim][row] += V^T[dim][token] . P[token][row]: the 16 tokens of the K step are the two
//           score n-tiles, so the B fragment is the lane's own score accumulators turned into
//           probabilities; the rows (dims) are permuted so that a lane's slice of a value row is D/8
//           contiguous dims, and each A register pairs two tokens of one dim (one byte permute).
//           P goes in as a high and a low part in the input type (two MMAs), so the probabilities
//           carry about 2^-17 relative error instead of the type's own rounding.
constexpr int kSmWarps = 4;
constexpr int kSmThreads = 32 * kSmWarps;

template <bool BF16>
__device__ __forceinline__ void mma_m16n8k16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint32_t b0, uint32_t b1) {
    if constexpr (BF16) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    } else {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
}

// two floats -> one register of the input type (round to nearest), and back
template <bool BF16>
__device__ __forceinline__ uint32_t pack_rn(float lo, float hi) {
    if constexpr (BF16) {
        const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&v);
    } else {
        const __half2 v = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&v);
    }
}
template <bool BF16>
__device__ __forceinline__ float2 unpack2(uint32_t w) {
    if constexpr (BF16) return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
    else return __half22float2(*reinterpret_cast<const __half2*>(&w));
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
    return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}
__device__ __forceinline__ float ex2a(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// One 16-token step (tokens tb .. tb + 15 of one unit's [token][D] key and value rows) of the warp-level
// MMA attention of up to 8 query rows: loads of tokens < n_tok, scores of this lane's row g, the online
// softmax update of (m, l) over the tokens the row sees (token < lim), and the value accumulation into o
// (rows 2t and 2t + 1). The first step a row takes must contain a token it sees.
template <int D, bool BF16>
__device__ __forceinline__ void mma_step(const uint16_t* __restrict__ kb, const uint16_t* __restrict__ vb, int64_t tb,
                                         int64_t n_tok, int64_t lim, float scale_log2, const uint32_t (&qa)[D / 16][2],
                                         float& m, float& l, float (&o)[D / 16][4], int g, int t) {
    constexpr int KS = D / 16;   // score k-steps
    constexpr int DPT = D / 4;   // key dims per lane quad position
    constexpr int DV = D / 8;    // value dims per lane group row
    constexpr int MT = D / 16;   // value m-tiles
    constexpr int KC = DPT / 8;  // 16-byte key chunks per lane and token
    constexpr int VC = DV / 8;   // 16-byte value chunks per lane and token
    // keys of tokens tb + 8 jj + g (score n-tile jj, column g): dims DPT t .. DPT t + DPT
    uint4 kw[2][KC];
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
        const int64_t tok = tb + 8 * jj + g;
        const uint4* kp = reinterpret_cast<const uint4*>(kb + tok * D + DPT * t);
#pragma unroll
        for (int c = 0; c < KC; ++c) kw[jj][c] = tok < n_tok ? __ldg(kp + c) : make_uint4(0u, 0u, 0u, 0u);
    }
    // values of tokens tb + {2t, 2t + 1, 8 + 2t, 9 + 2t} (value k = 2t, 2t+1, 2t+8, 2t+9): dims DV g ..
    uint4 vw[4][VC];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int64_t tok = tb + (e >> 1) * 8 + 2 * t + (e & 1);
        const uint4* vp = reinterpret_cast<const uint4*>(vb + tok * D + DV * g);
#pragma unroll
        for (int c = 0; c < VC; ++c) vw[e][c] = tok < n_tok ? __ldg(vp + c) : make_uint4(0u, 0u, 0u, 0u);
    }
    // scores of row g for tokens tb + 8 jj + 2t + {0, 1}
    float sc[2][4];
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
        sc[jj][0] = sc[jj][1] = sc[jj][2] = sc[jj][3] = 0.0f;
#pragma unroll
        for (int s = 0; s < KS; ++s)
            mma_m16n8k16<BF16>(sc[jj], qa[s][0], 0u, qa[s][1], 0u, word_of(kw[jj][s >> 1], 2 * (s & 1)),
                               word_of(kw[jj][s >> 1], 2 * (s & 1) + 1));
    }
    float x[2][2];
    float mx = -INFINITY;
#pragma unroll
    for (int jj = 0; jj < 2; ++jj)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int64_t tok = tb + 8 * jj + 2 * t + e;
            x[jj][e] = tok < lim ? sc[jj][e] * scale_log2 : -INFINITY;
            mx = fmaxf(mx, x[jj][e]);
        }
    // a row sees token 0 at its first step, so m is finite from then on; a later step whose tokens the
    // row cannot see leaves m unchanged (mx = -inf) and adds p = 0
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float mn = fmaxf(m, mx);
    const bool raise = mn > m;
    const float alpha = ex2a(m - mn);   // 0 at the first step (m = -inf), 1 when the max holds
    m = mn;
    float p[2][2];
    float ps = 0.0f;
#pragma unroll
    for (int jj = 0; jj < 2; ++jj)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            p[jj][e] = ex2a(x[jj][e] - mn);
            ps += p[jj][e];
        }
    l = l * alpha + ps;
    if (__any_sync(0xffffffffu, raise)) {
        // accumulator rows 2t and 2t + 1 belong to lane quads 2t and 2t + 1
        const float a0 = __shfl_sync(0xffffffffu, alpha, 8 * t);
        const float a1 = __shfl_sync(0xffffffffu, alpha, 8 * t + 4);
#pragma unroll
        for (int i = 0; i < MT; ++i) {
            o[i][0] *= a0;
            o[i][1] *= a1;
            o[i][2] *= a0;
            o[i][3] *= a1;
        }
    }
    // B fragments: k = 2t, 2t+1 are this lane's n-tile 0 columns, k = 2t+8, 2t+9 its n-tile 1 columns
    const uint32_t bh0 = pack_rn<BF16>(p[0][0], p[0][1]), bh1 = pack_rn<BF16>(p[1][0], p[1][1]);
    const float2 f0 = unpack2<BF16>(bh0), f1 = unpack2<BF16>(bh1);
    const uint32_t bl0 = pack_rn<BF16>(p[0][0] - f0.x, p[0][1] - f0.y);
    const uint32_t bl1 = pack_rn<BF16>(p[1][0] - f1.x, p[1][1] - f1.y);
    // m-tile i: A rows g and g + 8 are dims DV g + 2i and DV g + 2i + 1, i.e. the low and high
    // halves of word i of each token's slice
#pragma unroll
    for (int i = 0; i < MT; ++i) {
        const uint32_t w0 = word_of(vw[0][i >> 2], i & 3), w1 = word_of(vw[1][i >> 2], i & 3);
        const uint32_t w2 = word_of(vw[2][i >> 2], i & 3), w3 = word_of(vw[3][i >> 2], i & 3);
        const uint32_t a0 = prmt(w0, w1, 0x5410u), a1 = prmt(w0, w1, 0x7632u);
        const uint32_t a2 = prmt(w2, w3, 0x5410u), a3 = prmt(w2, w3, 0x7632u);
        mma_m16n8k16<BF16>(o[i], a0, a1, a2, a3, bh0, bh1);
        mma_m16n8k16<BF16>(o[i], a0, a1, a2, a3, bl0, bl1);
    }
}

// Query fragment of one row (row == nullptr: a zero padding row): k-step s takes the lane's words 2s
// (a0) and 2s + 1 (a2) of dims D/4 * t .. D/4 * t + D/4 - 1.
template <int D>
__device__ __forceinline__ void load_query_frag(const uint16_t* row, int t, uint32_t (&qa)[D / 16][2]) {
    constexpr int KC = D / 32;   // 16-byte chunks of the lane's quarter
    if (row) {
        const uint4* qp = reinterpret_cast<const uint4*>(row + (D / 4) * t);
#pragma unroll
        for (int c = 0; c < KC; ++c) {
            const uint4 w = __ldg(qp + c);
            qa[2 * c][0] = w.x;
            qa[2 * c][1] = w.y;
            qa[2 * c + 1][0] = w.z;
            qa[2 * c + 1][1] = w.w;
        }
    } else {
#pragma unroll
        for (int s = 0; s < D / 16; ++s) qa[s][0] = qa[s][1] = 0u;
    }
}

template <int D, bool BF16>
__global__ void __launch_bounds__(kSmThreads, 3) suffix_mma(const uint16_t* __restrict__ q,
                                                            const uint16_t* __restrict__ sk,
                                                            const uint16_t* __restrict__ sv, int H, int Hq, int64_t S,
                                                            int64_t n_units, float scale_log2,
                                                            float* __restrict__ acc_out, float* __restrict__ ml_out) {
    constexpr int KS = D / 16;   // score k-steps
    constexpr int DV = D / 8;    // value dims per lane group row
    constexpr int MT = D / 16;   // value m-tiles
    __shared__ __align__(16) float pacc[kSmWarps][8][D];
    __shared__ float pm[kSmWarps][8], pl[kSmWarps][8];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
    const int G = Hq / H;
    const int64_t nsteps = (S + 15) / 16;
    const int64_t s0 = warp * nsteps / kSmWarps, s1 = (warp + 1) * nsteps / kSmWarps;

    for (int64_t unit = blockIdx.x; unit < n_units; unit += gridDim.x) {
        const int64_t la = unit / H;   // layer * A + agent
        const int h = (int)(unit - la * H);
        const uint16_t* kb = sk + unit * S * D;
        const uint16_t* vb = sv + unit * S * D;
        uint32_t qa[KS][2];
        load_query_frag<D>(g < G ? q + ((la * Hq) + h * G + g) * D : nullptr, t, qa);
        float m = -INFINITY, l = 0.0f;
        float o[MT][4];
#pragma unroll
        for (int i = 0; i < MT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;

        for (int64_t st = s0; st < s1; ++st)
            mma_step<D, BF16>(kb, vb, st * 16, S, S, scale_log2, qa, m, l, o, g, t);
        l += __shfl_xor_sync(0xffffffffu, l, 1);
        l += __shfl_xor_sync(0xffffffffu, l, 2);
        // this warp's partial: o[i] holds rows 2t, 2t+1 at dims DV g + 2i (0, 1) and DV g + 2i + 1 (2, 3)
#pragma unroll
        for (int i = 0; i < MT; ++i) {
            pacc[warp][2 * t][DV * g + 2 * i] = o[i][0];
            pacc[warp][2 * t + 1][DV * g + 2 * i] = o[i][1];
            pacc[warp][2 * t][DV * g + 2 * i + 1] = o[i][2];
            pacc[warp][2 * t + 1][DV * g + 2 * i + 1] = o[i][3];
        }
        if (t == 0) {
            pm[warp][g] = m;   // -inf for a warp with no tokens of this unit
            pl[warp][g] = l;
        }
        __syncthreads();
        for (int idx = tid; idx < G * D; idx += kSmThreads) {
            const int r = idx / D, col = idx - r * D;
            float M = pm[0][r];
#pragma unroll
            for (int w = 1; w < kSmWarps; ++w) M = fmaxf(M, pm[w][r]);
            float sum = 0.0f;
#pragma unroll
            for (int w = 0; w < kSmWarps; ++w)
                if (pm[w][r] != -INFINITY) sum += pacc[w][r][col] * ex2a(pm[w][r] - M);
            acc_out[((la * Hq) + h * G + r) * D + col] = sum;
        }
        if (tid < G) {
            float M = pm[0][tid];
#pragma unroll
            for (int w = 1; w < kSmWarps; ++w) M = fmaxf(M, pm[w][tid]);
            float L = 0.0f;
#pragma unroll
            for (int w = 0; w < kSmWarps; ++w)
                if (pm[w][tid] != -INFINITY) L += pl[w][tid] * ex2a(pm[w][tid] - M);
            ml_out[((la * Hq) + h * G + tid) * 2] = M;
            ml_out[((la * Hq) + h * G + tid) * 2 + 1] = L;
        }
        __syncthreads();   // the partials' shared memory is reused by the next unit
    }
}

// ---------------------------------------------------------------- query-chunk mode on warp-level MMAs
// The causal part of query-chunk mode (G <= 8): query row r = c G + g of a (layer, agent, kv head) unit
// (chunk position c, query head g) sees the unit's chunk tokens 0..c. One warp takes 8 consecutive rows of
// one unit at a time (a task; tasks of one unit are consecutive, so its chunk keys and values are read
// from HBM once and then from L2) and runs mma_step over 16-token steps up to its last row's position,
// each row masked at its own position. Each row's partial (running max in log2 units, sum, unnormalised
// accumulator in the original basis) goes to the suffix slot of virtual agent a C + c.
template <int D, bool BF16>
__global__ void __launch_bounds__(kSmThreads, 3) chunk_mma(const uint16_t* __restrict__ q,
                                                           const uint16_t* __restrict__ ck,
                                                           const uint16_t* __restrict__ cv, int H, int Hq, int64_t C,
                                                           int64_t n_units, float scale_log2,
                                                           float* __restrict__ acc_out, float* __restrict__ ml_out) {
    constexpr int KS = D / 16;
    constexpr int DV = D / 8;
    constexpr int MT = D / 16;
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int G = Hq / H;
    const int64_t rows = C * G;
    const int64_t nrb = (rows + 7) / 8;
    const int64_t tasks = n_units * nrb;
    for (int64_t task = (int64_t)blockIdx.x * kSmWarps + (threadIdx.x >> 5); task < tasks;
         task += (int64_t)gridDim.x * kSmWarps) {
        const int64_t u = task / nrb, rb = task - u * nrb;
        const int64_t la = u / H;   // layer * A + agent
        const int h = (int)(u - la * H);
        const uint16_t* kb = ck + u * C * D;
        const uint16_t* vb = cv + u * C * D;
        // this lane's score row rb * 8 + g: position c_row sees tokens 0..c_row
        const int64_t row = rb * 8 + g;
        const bool real = row < rows;
        const int64_t c_row = real ? row / G : 0;
        uint32_t qa[KS][2];
        load_query_frag<D>(real ? q + ((la * C + c_row) * Hq + h * G + (row - c_row * G)) * D : nullptr, t, qa);
        const int64_t last_row = (rb * 8 + 7 < rows ? rb * 8 + 7 : rows - 1);
        const int64_t nsteps = last_row / G / 16 + 1;
        float m = -INFINITY, l = 0.0f;
        float o[MT][4];
#pragma unroll
        for (int i = 0; i < MT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;
        for (int64_t st = 0; st < nsteps; ++st)
            mma_step<D, BF16>(kb, vb, st * 16, C, c_row + 1, scale_log2, qa, m, l, o, g, t);
        l += __shfl_xor_sync(0xffffffffu, l, 1);
        l += __shfl_xor_sync(0xffffffffu, l, 2);
        // o[i] holds rows 2t (0, 2) and 2t + 1 (1, 3) at dims DV g + 2i (0, 1) and DV g + 2i + 1 (2, 3)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int64_t ro = rb * 8 + 2 * t + e;
            if (ro < rows) {
                const int64_t co = ro / G;
                float* dst = acc_out + ((la * C + co) * Hq + h * G + (ro - co * G)) * D + DV * g;
#pragma unroll
                for (int i = 0; i < MT; ++i)
                    *reinterpret_cast<float2*>(dst + 2 * i) = make_float2(o[i][e], o[i][2 + e]);
            }
        }
        if (t == 0 && real) {
            const int64_t orow = (la * C + c_row) * Hq + h * G + (row - c_row * G);
            ml_out[orow * 2] = m;
            ml_out[orow * 2 + 1] = l;
        }
    }
}

// ---------------------------------------------------------------- query-chunk mode
// Each agent's chunk of C query tokens carries its own keys/values; query token c sees the agent's
// chunk tokens 0..c (plus the pool, merged later). One block per (layer, agent, kv head, block of 32
// query rows r = c * G + g); chunk keys/values go through shared memory in tiles of 64 tokens; one
// warp owns 8 rows (one online-softmax state each), a lane one token of the tile for the scores and
// D/32 head dims for the accumulator. The partial (running max in log2 units, sum, unnormalised
// accumulator in the original basis) goes to the same slots as a suffix partial, with the chunk
// position folded into the agent index (a' = a * C + c).
constexpr int kChT = 64;
constexpr int kChRows = 32;
constexpr int kChThreads = 128;

template <int D>
constexpr size_t chunk_smem_bytes() {
    return sizeof(float) * ((size_t)kChT * (D + 1) + (size_t)kChT * D + (size_t)kChRows * D + 4 * kChT);
}

template <int D, bool BF16>
__global__ void __launch_bounds__(kChThreads) chunk_partial(const uint16_t* __restrict__ q,
                                                            const uint16_t* __restrict__ ck,
                                                            const uint16_t* __restrict__ cv, int H, int Hq, int64_t C,
                                                            float scale_log2, float* __restrict__ acc_out,
                                                            float* __restrict__ ml_out) {
    extern __shared__ float chs[];
    float* Ks = chs;                       // [kChT][D + 1]
    float* Vs = Ks + kChT * (D + 1);       // [kChT][D]
    float* Qs = Vs + kChT * D;             // [kChRows][D]
    float* Ps = Qs + kChRows * D;          // [4 warps][kChT]
    constexpr int RW = kChRows / 4;        // rows per warp
    constexpr int DPL = D / 32;            // accumulator dims per lane
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = Hq / H;
    const int64_t unit = blockIdx.x;       // (layer * A + a) * H + h
    const int h = (int)(unit % H);
    const int64_t la = unit / H;           // layer * A + a
    const int64_t rows = C * G;
    const int64_t r0 = (int64_t)blockIdx.y * kChRows;
    const uint16_t* kb = ck + unit * C * D;
    const uint16_t* vb = cv + unit * C * D;

    for (int i = tid; i < kChRows * D; i += kChThreads) {
        const int64_t r = r0 + i / D;
        float x = 0.0f;
        if (r < rows) {
            const int64_t c = r / G;
            const int g = (int)(r % G);
            x = bits_to_float(q[((la * C + c) * Hq + h * G + g) * D + i % D], BF16);
        }
        Qs[i] = x;
    }
    float m[RW], l[RW], acc[RW][DPL];
#pragma unroll
    for (int i = 0; i < RW; ++i) {
        m[i] = -INFINITY;
        l[i] = 0.0f;
#pragma unroll
        for (int e = 0; e < DPL; ++e) acc[i][e] = 0.0f;
    }
    const int64_t r_last = (r0 + kChRows < rows ? r0 + kChRows : rows) - 1;
    const int64_t c_max = r_last / G;
    for (int64_t t0 = 0; t0 <= c_max; t0 += kChT) {
        __syncthreads();
        for (int i = tid; i < kChT * D; i += kChThreads) {
            const int tk = i / D, dd = i % D;
            const bool ok = t0 + tk < C;
            Ks[tk * (D + 1) + dd] = ok ? bits_to_float(kb[(t0 + tk) * D + dd], BF16) : 0.0f;
            Vs[tk * D + dd] = ok ? bits_to_float(vb[(t0 + tk) * D + dd], BF16) : 0.0f;
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < RW; ++i) {
            const int ri = warp * RW + i;
            const int64_t r = r0 + ri;
            if (r >= rows) continue;               // warp-uniform
            const int64_t c = r / G;
            if (t0 > c) continue;                  // no visible token in this tile (warp-uniform)
            const float* qr = Qs + ri * D;
            float x0 = 0.0f, x1 = 0.0f;
#pragma unroll 8
            for (int dd = 0; dd < D; ++dd) {
                x0 = fmaf(qr[dd], Ks[lane * (D + 1) + dd], x0);
                x1 = fmaf(qr[dd], Ks[(lane + 32) * (D + 1) + dd], x1);
            }
            x0 = (t0 + lane <= c) ? x0 * scale_log2 : -INFINITY;
            x1 = (t0 + lane + 32 <= c) ? x1 * scale_log2 : -INFINITY;
            float tmax = fmaxf(x0, x1);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
            const float mn = fmaxf(m[i], tmax);
            const float alpha = m[i] == -INFINITY ? 0.0f : exp2f(m[i] - mn);
            const float p0 = exp2f(x0 - mn), p1 = exp2f(x1 - mn);
            float ps = p0 + p1;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
            l[i] = l[i] * alpha + ps;
            m[i] = mn;
            Ps[warp * kChT + lane] = p0;
            Ps[warp * kChT + lane + 32] = p1;
            __syncwarp();
#pragma unroll
            for (int e = 0; e < DPL; ++e) acc[i][e] *= alpha;
            const int tmaxk = (int)((c - t0 + 1) < kChT ? (c - t0 + 1) : kChT);
            for (int tk = 0; tk < tmaxk; ++tk) {
                const float pp = Ps[warp * kChT + tk];
#pragma unroll
                for (int e = 0; e < DPL; ++e) acc[i][e] = fmaf(pp, Vs[tk * D + lane * DPL + e], acc[i][e]);
            }
            __syncwarp();
        }
    }
#pragma unroll
    for (int i = 0; i < RW; ++i) {
        const int64_t r = r0 + warp * RW + i;
        if (r >= rows) continue;
        const int64_t c = r / G;
        const int g = (int)(r % G);
        const int64_t orow = (la * C + c) * Hq + h * G + g;
#pragma unroll
        for (int e = 0; e < DPL; ++e) acc_out[orow * D + lane * DPL + e] = acc[i][e];
        if (lane == 0) {
            ml_out[orow * 2] = m[i];
            ml_out[orow * 2 + 1] = l[i];
        }
    }
}

template <int D, bool BF16>
polykv_status launch_chunk_mma(const SuffixArgs& a, int L, int A_virtual, int H, int Hq, float sl, cudaStream_t st);

template <int D, bool BF16>
polykv_status run_chunk(const SuffixArgs& a, int L, int A_virtual, int H, int Hq, float scale, cudaStream_t st) {
    const int G = Hq / H;
    const int64_t C = a.chunk;
    // up to 8 query heads per kv head on the warp-level MMAs; more on the CUDA-core kernel
    if (G <= 8) return launch_chunk_mma<D, BF16>(a, L, A_virtual, H, Hq, scale * 1.4426950408889634f, st);
    const int64_t A = A_virtual / C;
    const int64_t nblk_rows = (C * G + kChRows - 1) / kChRows;
    if (nblk_rows > 65535) return set_error(POLYKV_E_UNSUPPORTED, "chunk: %lld query rows per kv head", (long long)(C * G));
    const dim3 grid((unsigned)((int64_t)L * A * H), (unsigned)nblk_rows);
    constexpr size_t smem = chunk_smem_bytes<D>();
    cudaError_t e = cudaFuncSetAttribute(chunk_partial<D, BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return set_error(POLYKV_E_CUDA, "chunk: smem attribute: %s", cudaGetErrorString(e));
    chunk_partial<D, BF16><<<grid, kChThreads, smem, st>>>(
        static_cast<const uint16_t*>(a.q), static_cast<const uint16_t*>(a.k), static_cast<const uint16_t*>(a.v), H, Hq,
        C, scale * 1.4426950408889634f, a.acc, a.ml);
    e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(POLYKV_E_CUDA, "chunk launch: %s", cudaGetErrorString(e));
    return POLYKV_OK;
}

template <int D, bool BF16>
polykv_status launch_chunk_mma(const SuffixArgs& a, int L, int A_virtual, int H, int Hq, float sl, cudaStream_t st) {
    auto kern = chunk_mma<D, BF16>;
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kSmThreads, 0);
    if (e != cudaSuccess || per_sm < 1) per_sm = 1;
    const int64_t C = a.chunk;
    const int64_t units = (int64_t)L * (A_virtual / C) * H;
    const int64_t tasks = units * ((C * (Hq / H) + 7) / 8);
    const int64_t need = (tasks + kSmWarps - 1) / kSmWarps;
    const int64_t cap = (int64_t)device_sm_count() * per_sm;
    const unsigned blocks = (unsigned)(need < cap ? need : cap);
    kern<<<blocks, kSmThreads, 0, st>>>(static_cast<const uint16_t*>(a.q), static_cast<const uint16_t*>(a.k),
                                        static_cast<const uint16_t*>(a.v), H, Hq, C, units, sl, a.acc, a.ml);
    e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(POLYKV_E_CUDA, "chunk launch: %s", cudaGetErrorString(e));
    return POLYKV_OK;
}

template <int D, int GMAX, bool BF16>
polykv_status launch_suffix_partial(const SuffixArgs& a, int L, int A, int H, int Hq, float sl, cudaStream_t st) {
    constexpr int smem = SfxTileSmem<D>::kBytes;
    auto kern = suffix_partial<D, GMAX, BF16>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return set_error(POLYKV_E_CUDA, "suffix: smem attribute: %s", cudaGetErrorString(e));
    const unsigned blocks = (unsigned)((int64_t)L * A * H);
    kern<<<blocks, kSfxThreads, smem, st>>>(static_cast<const uint16_t*>(a.q), static_cast<const uint16_t*>(a.k),
                                            static_cast<const uint16_t*>(a.v), A, H, Hq, a.len, sl, a.acc, a.ml);
    e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(POLYKV_E_CUDA, "suffix launch: %s", cudaGetErrorString(e));
    return POLYKV_OK;
}

template <int D, bool BF16>
polykv_status launch_suffix_mma(const SuffixArgs& a, int L, int A, int H, int Hq, float sl, cudaStream_t st) {
    auto kern = suffix_mma<D, BF16>;
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kSmThreads, 0);
    if (e != cudaSuccess || per_sm < 1) per_sm = 1;
    const int64_t units = (int64_t)L * A * H;
    const int64_t cap = (int64_t)device_sm_count() * per_sm;
    const unsigned blocks = (unsigned)(units < cap ? units : cap);
    kern<<<blocks, kSmThreads, 0, st>>>(static_cast<const uint16_t*>(a.q), static_cast<const uint16_t*>(a.k),
                                        static_cast<const uint16_t*>(a.v), H, Hq, a.len, units, sl, a.acc, a.ml);
    e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(POLYKV_E_CUDA, "suffix launch: %s", cudaGetErrorString(e));
    return POLYKV_OK;
}

template <int D, bool BF16>
polykv_status run_suffix(const SuffixArgs& a, int L, int A, int H, int Hq, float scale, cudaStream_t st) {
    const int G = Hq / H;
    const float sl = scale * 1.4426950408889634f;
    if (a.len < 1) return set_error(POLYKV_E_INVAL, "suffix: length %lld", (long long)a.len);
    // up to 8 query rows per kv head on the warp-level MMAs; more rows on the CUDA-core kernel
    if (G <= 8) return launch_suffix_mma<D, BF16>(a, L, A, H, Hq, sl, st);
    return launch_suffix_partial<D, 16, BF16>(a, L, A, H, Hq, sl, st);
}

}  // namespace

polykv_status launch_attend_suffix(const SuffixArgs& a, polykv_dtype dt, int L, int A, int H, int Hq, int D,
                                   float scale, cudaStream_t st) {
    const bool bf = dt == POLYKV_BF16;
    if (a.chunk > 0) {
        if (D == 128) return bf ? run_chunk<128, true>(a, L, A, H, Hq, scale, st) : run_chunk<128, false>(a, L, A, H, Hq, scale, st);
        if (D == 64) return bf ? run_chunk<64, true>(a, L, A, H, Hq, scale, st) : run_chunk<64, false>(a, L, A, H, Hq, scale, st);
        return set_error(POLYKV_E_UNSUPPORTED, "chunk: head_dim %d", D);
    }
    if (D == 128) return bf ? run_suffix<128, true>(a, L, A, H, Hq, scale, st) : run_suffix<128, false>(a, L, A, H, Hq, scale, st);
    if (D == 64) return bf ? run_suffix<64, true>(a, L, A, H, Hq, scale, st) : run_suffix<64, false>(a, L, A, H, Hq, scale, st);
    return set_error(POLYKV_E_UNSUPPORTED, "suffix: head_dim %d", D);
}

}  // namespace polykv
