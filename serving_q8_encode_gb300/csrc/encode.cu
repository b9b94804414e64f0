// Encode kernel: writes the shared pool (keys -> q8_0, values -> FWHT + 3-bit codes).
//
// PolyKV abstract ("PolyKV: A Shared Asymmetrically-Compressed KV Cache Pool
// for Multi-Agent LLM Inference"): keys int8 q8_0, values FWHT rotation then
// 3-bit Lloyd-Max quantization tuned to N(0,1), written once.
//
// Work mapping: one block of d threads per (unit, group of 32 consecutive pool
// tokens). Phase 1: d/32 lanes own one token; each lane holds one whole
// 32-element q8_0 block of the key and 32 consecutive value coordinates (four
// 16-byte loads each), writes the key codes and scale, and leaves the rotated
// value coordinates in shared memory. Phase 2: thread j decides the 32 tokens'
// codes of coordinate j and writes them as the pool's 12-byte string (token k
// at bits 3k..3k+2). The fp32 operation order is fixed (the CPU oracle
// restates it):
//   keys:   amax over the block; s16 = fp16_rn(amax / 127) (IEEE division);
//           code = round-half-away(x / s16), the quotient correctly rounded;
//   values: ||v||^2 = per 8-coordinate group a left-to-right sum of rounded
//           squares, then a pairwise tree over the d/8 group sums (two levels
//           inside the lane, the rest by xor-shuffles); FWHT butterflies at
//           strides 1..16 inside the lane and 32, 64 across lanes, each
//           (a, b) -> (a + b, a - b) with a the lower index; u = y / ||v||;
//           code = number of boundaries <= u.
// Neither decision needs the quotient itself:
//   keys:   x (bf16/fp16) and s16 have short significands, so x / s16 is either
//           exactly a half-integer or at least 2^-13 away from every
//           half-integer (x and s16 are small odd integers times powers of
//           two). With a normal scale the code is the integer nearest to
//           x * yb, yb a hair above 1 / s16, read from the mantissa of one
//           fused multiply-add (details at the key step); a zero, subnormal or
//           non-finite scale takes a slower path with the [-127, 127] clamp;
//   values: u >= b  <=>  y >= b * ||v|| except when u is within a few ulps of b
//           (where the rounding of either side can flip the comparison); such
//           boundary cases are the only ones allowed to differ from the
//           definition (they lie within 1e-6 relative of a boundary).
// Pairs of fp32 lanes use Blackwell's packed f32x2 add/mul/fma, which round
// each element exactly like the scalar instructions.
#include <cstring>

#include "polykv_internal.cuh"

namespace polykv {
namespace {

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
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f2u(a)), "l"(f2u(b)));
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

__device__ __forceinline__ void fetch32(const uint16_t* src, uint4 (&raw)[4]) {
    const uint4* p = reinterpret_cast<const uint4*>(src);
#pragma unroll
    for (int c = 0; c < 4; ++c) raw[c] = __ldcs(p + c);
}

__device__ __forceinline__ void unpack32(const uint4 (&raw)[4], float (&x)[32], bool bf16) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint32_t w[4] = {raw[c].x, raw[c].y, raw[c].z, raw[c].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (bf16) {
                x[8 * c + 2 * i] = __uint_as_float(w[i] << 16);
                x[8 * c + 2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
            } else {
                const __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
                const float2 f = __half22float2(h);
                x[8 * c + 2 * i] = f.x;
                x[8 * c + 2 * i + 1] = f.y;
            }
        }
    }
}

__device__ __forceinline__ float ge_f32(float a, float b) {
    float r;  // 1.0f if a >= b else 0.0f
    asm("set.ge.f32.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

// three-input maximum that returns NaN if any input is NaN (a block holding a NaN then gets a NaN
// scale and all-zero codes, as when the maximum is taken with NaN propagation)
__device__ __forceinline__ float max3(float a, float b, float c) {
    float r;
    asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// trunc(r + copysign(0.5 + 2^-14, r)) with the addition rounded toward zero = sign(r) * floor(|r| + 0.5 + 2^-14)
__device__ __forceinline__ int round_away(float r) {
    const float c = __uint_as_float((__float_as_uint(r) & 0x80000000u) | 0x3F000400u);   // +-(0.5 + 2^-14)
    return __float2int_rz(__fadd_rz(r, c));
}

__device__ __forceinline__ uint32_t bytes4(int a, int b, int c, int d) {
    // low bytes of four ints -> one word (a in byte 0)
    uint32_t ab, cd, w;
    asm("prmt.b32 %0, %1, %2, 0x0040;" : "=r"(ab) : "r"(a), "r"(b));
    asm("prmt.b32 %0, %1, %2, 0x0040;" : "=r"(cd) : "r"(c), "r"(d));
    asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(w) : "r"(ab), "r"(cd));
    return w;
}

// One block of D threads per (unit, 32-token group) inside [t0, t0 + n). Phase 1: d/32 lanes per
// token (token tau = lane group, quarter gl) do the keys, the value norm, FWHT and 3-bit decisions,
// and leave the signed half-codes in shared memory. Phase 2: thread j = coordinate j packs the 32
// tokens' codes of coordinate j into its 12-byte string (token k at bits 3k..3k+2). Tokens of a partly covered group that lie outside [t0, t0 + n) keep
// the bits already in the pool.
template <int D>
struct EncSmem {
    static constexpr int kRow = D + 4;   // padded row of y (floats); chunks rotated, see enc_phys
    float y[32][kRow];                   // per token: the signed half-codes of its coordinates
};

// physical float index of coordinate j inside a row of EncSmem::y: 16-byte chunk c of lane quarter gl
// is stored at chunk (c + (256 / D) gl) mod 8 of that quarter; with the 4-float row padding, the
// lanes of one 8-lane store phase (8 / (D / 32) tokens x D / 32 quarters) land on distinct banks
template <int D>
__device__ __forceinline__ int enc_phys(int j) {
    const int gl = j >> 5, c = (j >> 2) & 7;
    return (gl << 5) | (((c + (256 / D) * gl) & 7) << 2) | (j & 3);
}

template <int D, bool BF16>
__global__ void __launch_bounds__(D, D == 128 ? 8 : 12) encode_kernel(const uint16_t* __restrict__ k,
                                                           const uint16_t* __restrict__ v, PoolView p,
                                                           int64_t n_tok, int64_t t0, int g_first, int n_groups) {
    constexpr int LPV = D / 32;          // lanes per token in phase 1
    __shared__ EncSmem<D> sm;
    const int tid = threadIdx.x;
    const int gl = tid % LPV;
    const int tau = tid / LPV;           // token of the group, 0..31
    const int64_t unit = blockIdx.x / n_groups;
    const int64_t grp = g_first + (int64_t)(blockIdx.x % n_groups);
    const int64_t tk = grp * 32 + tau;   // pool token
    const bool valid = tk >= t0 && tk < t0 + n_tok;
    const int64_t vi = unit * n_tok + (valid ? tk - t0 : 0);   // input row (row 0 of the unit if not valid)
    const int64_t pidx = unit * p.cap + tk;

    // both 64-byte rows are requested before any arithmetic (one memory round trip per lane)
    uint4 kraw[4], vraw[4];
    fetch32(k + vi * D + gl * 32, kraw);
    fetch32(v + vi * D + gl * 32, vraw);

    // ---------------- keys: one q8_0 block per lane
    {
        float x[32];
        unpack32(kraw, x, BF16);
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 32; i += 2) amax = max3(amax, fabsf(x[i]), fabsf(x[i + 1]));
        const __half s16 = __float2half_rn(__fdiv_rn(amax, 127.0f));
        const float sf = __half2float(s16);
        uint32_t packed[8];
        if (sf >= 6.103515625e-05f && sf <= 65504.0f) {
            // normal scale: the code is the integer nearest to x * yb, read from the low byte of
            // RN(x * yb + (2^23 + 256)), one fused multiply-add per element. yb is one ulp above
            // RU(1 / s16), so x * yb = (x / s16)(1 + e) with 0 < e <= 2^-22: an exact half-integer
            // quotient moves away from zero (ties away), and any other quotient, at least 2^-13 from
            // every half-integer, moves by at most 127.06 * 2^-22 < 2^-13 and keeps its nearest
            // integer. The sum lies in [2^23, 2^24), where RN rounds to an integer and the mantissa
            // holds 256 + code, whose low byte is the int8 code. |x / s16| <= 127.06: no clamp.
            const float yb = __uint_as_float(__float_as_uint(__frcp_ru(sf)) + 1u);
            const float2 yb2 = make_float2(yb, yb);
            const float2 mg2 = make_float2(8388864.0f, 8388864.0f);   // 2^23 + 256
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
                const float2 r01 = fma2(make_float2(x[i], x[i + 1]), yb2, mg2);
                const float2 r23 = fma2(make_float2(x[i + 2], x[i + 3]), yb2, mg2);
                packed[i >> 2] = bytes4(__float_as_int(r01.x), __float_as_int(r01.y), __float_as_int(r23.x),
                                        __float_as_int(r23.y));
            }
        } else {
            // zero, subnormal or non-finite scale: round half away from zero as
            // trunc(RN(x * RN(1/s16)) +- (0.5 + 2^-14)) with the addition rounded toward zero, then
            // the [-127, 127] clamp (a subnormal scale can take |x / s16| up to ~189); a scale that
            // is 0 or not finite gives y = 0 and all-zero codes
            const bool usable = sf > 0.0f && sf <= 65504.0f;
            const float yb = usable ? __frcp_rn(sf) : 0.0f;
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
                int q[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) q[e] = max(-127, min(127, round_away(__fmul_rn(x[i + e], yb))));
                packed[i >> 2] = bytes4(q[0], q[1], q[2], q[3]);
            }
        }
        if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(p.kq + pidx * D + gl * 32);
            dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
            dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
            p.ks[pidx * (D / kQ8Block) + gl] = s16;
        }
    }

    // ---------------- values, phase 1: norm and FWHT of this lane's quarter
    float y[32];
    unpack32(vraw, y, BF16);
    float nrm;
    {
        float2 sq[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) sq[i] = mul2(make_float2(y[2 * i], y[2 * i + 1]), make_float2(y[2 * i], y[2 * i + 1]));
        // groups g = 0..3 of 8 coordinates: group g's squares are sq[4g..4g+3] (.x, .y interleaved)
        // accumulate groups (0,1) and (2,3) as packed pairs, left to right inside each group
        float2 a01 = make_float2(sq[0].x, sq[4].x), a23 = make_float2(sq[8].x, sq[12].x);
        a01 = add2(a01, make_float2(sq[0].y, sq[4].y));
        a23 = add2(a23, make_float2(sq[8].y, sq[12].y));
#pragma unroll
        for (int e = 1; e < 4; ++e) {
            a01 = add2(a01, make_float2(sq[e].x, sq[4 + e].x));
            a23 = add2(a23, make_float2(sq[8 + e].x, sq[12 + e].x));
            a01 = add2(a01, make_float2(sq[e].y, sq[4 + e].y));
            a23 = add2(a23, make_float2(sq[8 + e].y, sq[12 + e].y));
        }
        float ss = __fadd_rn(__fadd_rn(a01.x, a01.y), __fadd_rn(a23.x, a23.y));
#pragma unroll
        for (int m = 1; m < LPV; m <<= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, m));
        nrm = __fsqrt_rn(ss);
    }
    // butterflies, stride 1 (scalar) then 2..16 (packed pairs)
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
        const float a = y[i], b = y[i + 1];
        y[i] = __fadd_rn(a, b);
        y[i + 1] = __fsub_rn(a, b);
    }
#pragma unroll
    for (int h = 2; h < 32; h <<= 1) {
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
            if ((i & h) == 0) {
                const float2 a = make_float2(y[i], y[i + 1]), b = make_float2(y[i + h], y[i + h + 1]);
                const float2 s = add2(a, b), d = sub2(a, b);
                y[i] = s.x;
                y[i + 1] = s.y;
                y[i + h] = d.x;
                y[i + h + 1] = d.y;
            }
        }
    }
#pragma unroll
    for (int m = 1; m < LPV; m <<= 1) {
        const float sg = (gl & m) ? -1.0f : 1.0f;  // upper lane: lower - upper; lower lane: lower + upper
        const float2 sg2 = make_float2(sg, sg);
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
            const float o0 = __shfl_xor_sync(0xffffffffu, y[i], m);
            const float o1 = __shfl_xor_sync(0xffffffffu, y[i + 1], m);
            const float2 r = fma2(sg2, make_float2(y[i], y[i + 1]), make_float2(o0, o1));
            y[i] = r.x;
            y[i + 1] = r.y;
        }
    }
    // code = number of boundaries b_i * ||v|| <= y. The boundaries are symmetric (b_{6-i} = -b_i,
    // b_3 = 0): with m = #{i in 4..6 : |y| >= t_i}, the code is 4 + m for y >= 0 and 3 - m for y < 0,
    // i.e. 3.5 + copysign(m + 0.5, y). The encoder keeps the signed half-code copysign(m + 0.5, y) = code - 3.5
    // as an exact float and adds the 3.5s of a whole group at once. For y < 0 the definition
    // compares |y| > t_i and y = -0 belongs to the upper half; both differences happen only at an exact
    // boundary (|y| equal to a scaled boundary, or u = 0), inside the boundary exemption. Float
    // arithmetic keeps this work on the FMA pipe; the integer/compare pipe is the encoder's bottleneck.
    // 3-bit decisions in registers: the signed half-code c - 3.5 of every coordinate, an exact float in
    // {+-0.5, +-1.5, +-2.5, +-3.5}; a zero norm gives u = 0 and code 4; a token outside [t0, t0 + n)
    // gets code 0 and keeps its old bits (phase 2)
    {
        const float t4 = __fmul_rn(kB4, nrm), t5 = __fmul_rn(kB5, nrm), t6 = __fmul_rn(kB6, nrm);
        if (valid && nrm > 0.0f) {
            // pairs of coordinates: the three 0/1 compares summed with packed adds (exact: small integers
            // and halves), then the sign of y
            const float2 half2 = make_float2(0.5f, 0.5f);
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
                const float a0 = fabsf(y[i]), a1 = fabsf(y[i + 1]);
                float2 h = add2(half2, make_float2(ge_f32(a0, t4), ge_f32(a1, t4)));
                h = add2(h, make_float2(ge_f32(a0, t5), ge_f32(a1, t5)));
                h = add2(h, make_float2(ge_f32(a0, t6), ge_f32(a1, t6)));
                y[i] = copysignf(h.x, y[i]);
                y[i + 1] = copysignf(h.y, y[i + 1]);
            }
        } else {
            // ||v|| = 0: every code is 4 (half-code 0.5); a token outside [t0, t0 + n): code 0 (-3.5), bits kept
            const float fv = valid ? 0.5f : -3.5f;
#pragma unroll
            for (int i = 0; i < 32; ++i) y[i] = fv;
        }
    }
    // the half-codes go to shared memory (rotated chunks, see enc_phys)
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        float4* dst = reinterpret_cast<float4*>(&sm.y[tau][enc_phys<D>(32 * gl + 4 * c)]);
        *dst = make_float4(y[4 * c], y[4 * c + 1], y[4 * c + 2], y[4 * c + 3]);
    }
    if (gl == 0 && valid) p.vn[pidx] = __float2half_rn(nrm);
    // running per-unit maximum of ||v|| (an upper bound used by attention to scale fp16 operands):
    // one max-reduction per warp, one atomic per warp. Norms are non-negative, so their bit patterns
    // order as unsigned integers.
    {
        const uint32_t nb = (gl == 0 && valid) ? __float_as_uint(nrm) : 0u;
        const uint32_t mx = __reduce_max_sync(0xffffffffu, nb);
        if ((tid & 31) == 0 && mx != 0u) atomicMax(reinterpret_cast<unsigned int*>(p.nmax) + unit, mx);
    }
    __syncthreads();

    // ---------------- values, phase 2: thread j = coordinate j packs the group's 32 codes
    {
        const int j = tid;
        const int pj = enc_phys<D>(j);
        const int64_t g0tok = grp * 32;
        const int kmin = (int)(t0 > g0tok ? t0 - g0tok : 0);                    // valid tokens: [kmin, kmax)
        const int kmax = (int)(t0 + n_tok - g0tok < 32 ? t0 + n_tok - g0tok : 32);
        // eight codes c_0..c_7 -> the 24-bit group sum c_i * 8^i, formed exactly in fp32: Horner over
        // the half-codes h_i = c_i - 3.5 gives sum h_i 8^i, a multiple of 1/2 below 2^23 in magnitude
        // (24 significant bits at most, so every step is exact); adding 3.5 * sum 8^i = 8388607.5
        // gives the integer group sum (< 2^24), also exactly.
        uint32_t w24[4];
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            float w = sm.y[8 * g + 7][pj];
#pragma unroll
            for (int i = 6; i >= 0; --i) w = fmaf(w, 8.0f, sm.y[8 * g + i][pj]);
            w24[g] = (uint32_t)__float2uint_rz(w + 8388607.5f);
        }
        uint32_t o0 = w24[0] | (w24[1] << 24);
        uint32_t o1 = (w24[1] >> 8) | (w24[2] << 16);
        uint32_t o2 = (w24[2] >> 16) | (w24[3] << 8);
        uint32_t* dst = reinterpret_cast<uint32_t*>(p.vc + ((unit * (p.cap / 32) + grp) * D + j) * 12);
        if (kmin > 0 || kmax < 32) {
            // a partly covered group keeps the other tokens' bits already in the pool
            const int lo = 3 * kmin, hi = 3 * kmax;   // new bits: [lo, hi) of the 96-bit string
            auto span = [](int a, int b) -> uint32_t {   // bits [a, b) of one 32-bit word, a, b clamped
                a = a < 0 ? 0 : (a > 32 ? 32 : a);
                b = b < 0 ? 0 : (b > 32 ? 32 : b);
                const uint32_t up = b >= 32 ? 0xFFFFFFFFu : ((1u << b) - 1u);
                const uint32_t dn = a >= 32 ? 0xFFFFFFFFu : ((1u << a) - 1u);
                return up & ~dn;
            };
            const uint32_t m0 = span(lo, hi), m1 = span(lo - 32, hi - 32), m2 = span(lo - 64, hi - 64);
            o0 = (dst[0] & ~m0) | (o0 & m0);
            o1 = (dst[1] & ~m1) | (o1 & m1);
            o2 = (dst[2] & ~m2) | (o2 & m2);
        }
        dst[0] = o0;
        dst[1] = o1;
        dst[2] = o2;
    }
}

template <int D, bool BF16>
polykv_status run(const PoolView& p, const void* k, const void* v, int64_t t0, int64_t n, cudaStream_t st) {
    const int64_t g_first = t0 / 32, g_last = (t0 + n - 1) / 32;
    const int64_t n_groups = g_last - g_first + 1;
    const int64_t blocks = (int64_t)p.L * p.H * n_groups;
    if (blocks > 0x7FFFFFFF || g_last > 0x7FFFFFFF)
        return set_error(POLYKV_E_UNSUPPORTED, "encode: too many token groups (%lld)", (long long)blocks);
    encode_kernel<D, BF16><<<(unsigned)blocks, D, 0, st>>>(static_cast<const uint16_t*>(k),
                                                           static_cast<const uint16_t*>(v), p, n, t0, (int)g_first,
                                                           (int)n_groups);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(POLYKV_E_CUDA, "encode launch: %s", cudaGetErrorString(e));
    return POLYKV_OK;
}

}  // namespace

polykv_status launch_encode(const PoolView& p, polykv_dtype dt, const void* k, const void* v, int64_t t0,
                            int64_t n_tokens, cudaStream_t stream) {
    const bool bf = dt == POLYKV_BF16;
    if (p.d == 128) return bf ? run<128, true>(p, k, v, t0, n_tokens, stream) : run<128, false>(p, k, v, t0, n_tokens, stream);
    if (p.d == 64) return bf ? run<64, true>(p, k, v, t0, n_tokens, stream) : run<64, false>(p, k, v, t0, n_tokens, stream);
    return set_error(POLYKV_E_UNSUPPORTED, "encode: head_dim %d", p.d);
}

}  // namespace polykv
