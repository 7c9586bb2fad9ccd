// attn_combine.cuh -- the combine kernel (step a7).
//
// minfer "10 · R4" §2.1/§3.2: per (sequence, query head), gmx = max over the
// splits of mx; each split is reweighted by w = exp(mx - gmx); S = sum w*S_sp,
// acc = sum w*oc_sp; o = acc / S, and 0 when S is 0 (every split empty). A
// split whose mx is -inf (no rows) gets weight 0 explicitly and its oc is never
// read, so an all-empty row gives o = 0 without evaluating -inf - (-inf).
// mx is in log2 units (the partial kernel folds log2 e into q), so the weights
// use the base-2 exponential.
#pragma once

#include "attn_device.cuh"

namespace attn {

template <int HD>
struct CombineCfg {
    static constexpr int THREADS = HD >= 256 ? 256 : 128;
    static constexpr int VEC = HD >= 4 ? 4 : HD;     // floats per thread per split row
    static constexpr int TPS = HD / VEC;             // threads per split row
    static constexpr int NG = THREADS / TPS;         // split groups summed in parallel
};

template <int HD>
__global__ void __launch_bounds__(CombineCfg<HD>::THREADS)
attn_combine(const CombineArgs a)
{
    using C = CombineCfg<HD>;
    extern __shared__ float sw[];                    // [P] weights, then [NG][HD] group sums
    __shared__ float red[32];
    __shared__ float bcast;

    pdl_wait();                                      // partials come from the previous grid

    const int h = blockIdx.x, s = blockIdx.y, tid = threadIdx.x;
    const int P = a.n_splits;
    const size_t row = (size_t)s * a.n_head + h;
    const float2 *ml = a.ws_ml + row * P;

    // gmx = max_sp mx_sp
    float mx = -INFINITY;
    for (int sp = tid; sp < P; sp += C::THREADS) mx = fmaxf(mx, ml[sp].x);
    mx = warp_max(mx);
    if ((tid & 31) == 0) red[tid >> 5] = mx;
    __syncthreads();
    if (tid == 0) {
        float t = red[0];
        for (int w = 1; w < C::THREADS / 32; ++w) t = fmaxf(t, red[w]);
        bcast = t;
    }
    __syncthreads();
    const float gmx = bcast;

    // w_sp and S = sum w * S_sp
    float S = 0.f;
    for (int sp = tid; sp < P; sp += C::THREADS) {
        const float2 v = ml[sp];
        const float w = (v.x == -INFINITY) ? 0.f : ex2(v.x - gmx);
        sw[sp] = w;
        S = fmaf(w, v.y, S);
    }
    S = warp_sum(S);
    __syncthreads();                                 // red[] reuse and sw[] visible
    if ((tid & 31) == 0) red[tid >> 5] = S;
    __syncthreads();
    if (tid == 0) {
        float t = 0.f;
        for (int w = 0; w < C::THREADS / 32; ++w) t += red[w];
        bcast = t;
    }

    // acc = sum w * oc_sp, split groups in parallel, then reduced
    const int grp = tid / C::TPS, dt = tid % C::TPS;
    float acc[C::VEC];
#pragma unroll
    for (int i = 0; i < C::VEC; ++i) acc[i] = 0.f;
    const float *oc = a.ws_o + row * P * HD + dt * C::VEC;
    for (int sp = grp; sp < P; sp += C::NG) {
        const float w = sw[sp];
        if (w != 0.f) {
            if constexpr (C::VEC == 4) {
                const float4 t = *reinterpret_cast<const float4 *>(oc + (size_t)sp * HD);
                acc[0] = fmaf(w, t.x, acc[0]); acc[1] = fmaf(w, t.y, acc[1]);
                acc[2] = fmaf(w, t.z, acc[2]); acc[3] = fmaf(w, t.w, acc[3]);
            } else {
#pragma unroll
                for (int i = 0; i < C::VEC; ++i) acc[i] = fmaf(w, oc[(size_t)sp * HD + i], acc[i]);
            }
        }
    }
    float *gs = sw + ((P + 3) & ~3);
#pragma unroll
    for (int i = 0; i < C::VEC; ++i) gs[grp * HD + dt * C::VEC + i] = acc[i];
    __syncthreads();
    const float Stot = bcast;
    for (int d = tid; d < HD; d += C::THREADS) {
        float t = 0.f;
        for (int g = 0; g < C::NG; ++g) t += gs[g * HD + d];
        a.out[row * HD + d] = Stot > 0.f ? t / Stot : 0.f;
    }
}

template <int HD>
constexpr size_t combine_smem_bytes(int n_splits)
{
    return (size_t)(((n_splits + 3) & ~3) + CombineCfg<HD>::NG * HD) * sizeof(float);
}

} // namespace attn
