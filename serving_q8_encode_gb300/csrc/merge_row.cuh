// Finishing one attention output row from merged partials: shared by the merge kernels and the
// warp-level attention kernel's in-kernel merge. Host code never includes this file.
#pragma once

#include <cmath>

#include "polykv_internal.cuh"

namespace polykv {

template <int D>
struct MergeVec;
template <>
struct MergeVec<128> {
    using T = float4;
    static __device__ __forceinline__ void to(const T& v, float* o) { o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w; }
    static __device__ __forceinline__ T from(const float* o) { return make_float4(o[0], o[1], o[2], o[3]); }
};
template <>
struct MergeVec<64> {
    using T = float2;
    static __device__ __forceinline__ void to(const T& v, float* o) { o[0] = v.x; o[1] = v.y; }
    static __device__ __forceinline__ T from(const float* o) { return make_float2(o[0], o[1]); }
};

// Finishes one output row from its merged rotated-basis accumulator o (this lane's D/32 elements),
// running maximum M and sum L: the inverse FWHT (1/D) H o, then the private suffix's partial (already
// in the original basis) under the same softmax, then the division by the total sum.
template <int D>
__device__ __forceinline__ void finish_row(float (&o)[D / 32], float M, float L, float2 sml,
                                           const typename MergeVec<D>::T& sv, int lane) {
    constexpr int EPL = D / 32;
    using V = MergeVec<D>;
    // in-lane butterflies (strides < EPL), then across lanes
#pragma unroll
    for (int h = 1; h < EPL; h <<= 1)
#pragma unroll
        for (int e = 0; e < EPL; ++e)
            if ((e & h) == 0) {
                const float x = o[e], y = o[e + h];
                o[e] = x + y;
                o[e + h] = x - y;
            }
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
            const float other = __shfl_xor_sync(0xffffffffu, o[e], m);
            o[e] = upper ? other - o[e] : o[e] + other;
        }
    }
#pragma unroll
    for (int e = 0; e < EPL; ++e) o[e] *= (1.0f / D);
    if (sml.x != -INFINITY) {
        // the suffix partial is already in the original basis
        const float Mn = fmaxf(M, sml.x);
        const float c = exp2f(M - Mn), w = exp2f(sml.x - Mn);
        float x[EPL];
        V::to(sv, x);
        L = fmaf(w, sml.y, L * c);
#pragma unroll
        for (int e = 0; e < EPL; ++e) o[e] = fmaf(w, x[e], o[e] * c);
    }
    const float inv = 1.0f / L;
#pragma unroll
    for (int e = 0; e < EPL; ++e) o[e] *= inv;
}

}  // namespace polykv
