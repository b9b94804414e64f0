// Encode kernel: writes the shared pool (keys -> q8_0, values -> FWHT + 3-bit codes).
//
// PolyKV abstract ("PolyKV: A Shared Asymmetrically-Compressed KV Cache Pool
// for Multi-Agent LLM Inference"): keys int8 q8_0, values FWHT rotation then
// 3-bit Lloyd-Max quantization tuned to N(0,1), written once.
//
// Work mapping: G = d/8 consecutive lanes own one (layer, kv head, token)
// position; each lane loads 8 key and 8 value elements with one 16-byte load
// each. The fp32 operation order below is fixed (the CPU oracle restates it):
//   keys:   block amax over 4 lanes (shuffle max), s16 = fp16_rn(amax / 127),
//           code = round-half-away(x / s16) with an IEEE division;
//   values: ||v||^2 = lane-local left-to-right sum of rounded squares, then an
//           xor-butterfly (pairwise tree) over the G lanes; FWHT butterflies at
//           strides 1, 2, 4 inside the lane and 8, 16, ... across lanes, each
//           (a, b) -> (a + b, a - b) with a the lower index; u = y / ||v||.
#include "polykv_internal.cuh"

namespace polykv {
namespace {

__device__ __forceinline__ void unpack8(const uint4 raw, float (&x)[8], bool bf16) {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t lo = w[i] & 0xFFFFu, hi = w[i] >> 16;
        if (bf16) {
            x[2 * i] = __uint_as_float(lo << 16);
            x[2 * i + 1] = __uint_as_float(hi << 16);
        } else {
            x[2 * i] = __half2float(__ushort_as_half((unsigned short)lo));
            x[2 * i + 1] = __half2float(__ushort_as_half((unsigned short)hi));
        }
    }
}

__device__ __forceinline__ uint32_t value_code(float u) {
    // number of boundaries b_i <= u, boundaries symmetric about 0
    const uint32_t c = (u >= -kB6) + (u >= -kB5) + (u >= -kB4) + (u >= 0.0f) + (u >= kB4) + (u >= kB5) +
                       (u >= kB6);
    return c;
}

template <int D, bool BF16>
__global__ void __launch_bounds__(256) encode_kernel(const uint16_t* __restrict__ k, const uint16_t* __restrict__ v,
                                                     PoolView p, int64_t n_tok, int64_t t0, int64_t n_vec) {
    constexpr int G = D / 8;             // lanes per vector
    constexpr int VPB = 256 / G;         // vectors per block
    const int gl = threadIdx.x % G;      // lane inside the vector group
    const int64_t vi_raw = (int64_t)blockIdx.x * VPB + threadIdx.x / G;
    const bool valid = vi_raw < n_vec;
    const int64_t vi = valid ? vi_raw : n_vec - 1;  // keep every lane in the shuffles
    const int64_t unit = vi / n_tok;
    const int64_t tok = t0 + (vi - unit * n_tok);
    const int64_t pidx = unit * p.cap + tok;        // pool position

    const uint4 kraw = __ldcs(reinterpret_cast<const uint4*>(k + vi * D) + gl);
    const uint4 vraw = __ldcs(reinterpret_cast<const uint4*>(v + vi * D) + gl);

    // ---------------- keys: q8_0
    float x[8];
    unpack8(kraw, x, BF16);
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(x[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const __half s16 = __float2half_rn(__fdiv_rn(amax, 127.0f));
    const float sf = __half2float(s16);
    const bool usable = sf > 0.0f && sf <= 65504.0f;
    uint32_t packed[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        int q = 0;
        if (usable) {
            const float r = __fdiv_rn(x[i], sf);
            q = (int)roundf(r);  // halfway cases away from zero
            q = max(-127, min(127, q));
        }
        packed[i >> 2] |= (uint32_t)(q & 0xFF) << (8 * (i & 3));
    }

    // ---------------- values: norm, FWHT, 3-bit codes
    float y[8];
    unpack8(vraw, y, BF16);
    float ss = __fmul_rn(y[0], y[0]);
#pragma unroll
    for (int i = 1; i < 8; ++i) ss = __fadd_rn(ss, __fmul_rn(y[i], y[i]));
#pragma unroll
    for (int m = 1; m < G; m <<= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, m));
    const float nrm = __fsqrt_rn(ss);

#pragma unroll
    for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if ((i & h) == 0) {
                const float a = y[i], b = y[i + h];
                y[i] = __fadd_rn(a, b);
                y[i + h] = __fsub_rn(a, b);
            }
        }
    }
#pragma unroll
    for (int m = 1; m < G; m <<= 1) {
        const bool upper = (gl & m) != 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float o = __shfl_xor_sync(0xffffffffu, y[i], m);
            y[i] = upper ? __fsub_rn(o, y[i]) : __fadd_rn(y[i], o);
        }
    }
    uint32_t w24 = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float u = nrm > 0.0f ? __fdiv_rn(y[i], nrm) : 0.0f;
        w24 |= value_code(u) << (3 * i);
    }
    // gather 3-byte lane words into 32-bit words: word j = bytes 4j..4j+3 of the vector's codes
    const int lo_lane = (4 * gl) / 3;
    const int shift = 8 * (4 * gl - 3 * lo_lane);
    const int grp_base = (threadIdx.x & 31) & ~(G - 1);
    const uint32_t wlo = __shfl_sync(0xffffffffu, w24, grp_base + min(lo_lane, G - 1));
    const uint32_t whi = __shfl_sync(0xffffffffu, w24, grp_base + min(lo_lane + 1, G - 1));
    const uint32_t word = (wlo >> shift) | (whi << (24 - shift));

    if (!valid) return;
    reinterpret_cast<uint2*>(p.kq + pidx * D)[gl] = make_uint2(packed[0], packed[1]);
    if ((gl & 3) == 0) p.ks[pidx * (D / kQ8Block) + gl / 4] = s16;
    if (gl < 3 * G / 4) reinterpret_cast<uint32_t*>(p.vc + pidx * (3 * D / 8))[gl] = word;
    if (gl == 0) p.vn[pidx] = __float2half_rn(nrm);
}

template <int D, bool BF16>
polykv_status run(const PoolView& p, const void* k, const void* v, int64_t t0, int64_t n, cudaStream_t st) {
    const int64_t n_vec = (int64_t)p.L * p.H * n;
    constexpr int VPB = 256 / (D / 8);
    const int64_t blocks = (n_vec + VPB - 1) / VPB;
    if (blocks > 0x7FFFFFFF) return set_error(POLYKV_E_UNSUPPORTED, "encode: too many vectors (%lld)", (long long)n_vec);
    encode_kernel<D, BF16><<<(unsigned)blocks, 256, 0, st>>>(static_cast<const uint16_t*>(k),
                                                              static_cast<const uint16_t*>(v), p, n, t0, n_vec);
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
