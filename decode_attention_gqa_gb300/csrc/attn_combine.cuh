// attn_combine.cuh -- the combine kernel (step a7).
//
// minfer "10 · R4" §2.1/§3.2: per (sequence, query head), gmx = max over the
// splits of mx; each split is reweighted by w = exp(mx - gmx); S = sum w*S_sp,
// acc = sum w*oc_sp; o = acc / S, and 0 when S is 0 (every split empty).
//
// Here the same merge is evaluated in one streaming pass so that every load of
// a block is issued up front: each warp folds its share of the splits into a
// running (m, S, acc) with the §2.1 update rule (a new maximum rescales what
// came before), then the warps' states are folded together the same way. The
// result equals the two-pass form up to rounding. A split whose mx is -inf
// (no rows) is skipped, so an all-empty row gives o = 0 without evaluating
// -inf - (-inf). mx is in log2 units (the partial kernel folds log2 e into q),
// so the weights use the base-2 exponential.
#pragma once

#include "attn_device.cuh"

namespace attn {

template <int HD>
struct CombineCfg {
    static constexpr int WARPS = 8;                   // split groups per head
    static constexpr int THREADS = WARPS * 32;
    static constexpr int VEC = HD >= 128 ? HD / 32 : 4;   // floats per lane per split row
    static constexpr int TPS = HD / VEC;              // lanes per split row
    static constexpr int LG = 32 / TPS;               // split rows per warp step
    static constexpr int BATCH = 8;                   // split rows in flight per lane
};

// Fold (m2, S2, a2) into (m, S, a): the §2.1 rescale-and-add rule.
template <int V>
__device__ __forceinline__ void fold(float &m, float &S, float (&acc)[V], float m2, float S2,
                                     const float (&a2)[V])
{
    if (m2 == -INFINITY) return;
    const float mn = fmaxf(m, m2);
    const float c1 = ex2(m - mn), c2 = ex2(m2 - mn);      // c1 = 0 while m = -inf
    S = S * c1 + S2 * c2;
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] = acc[i] * c1 + a2[i] * c2;
    m = mn;
}

template <int HD>
__global__ void __launch_bounds__(CombineCfg<HD>::THREADS)
attn_combine(const CombineArgs a)
{
    using C = CombineCfg<HD>;
    constexpr int V = C::VEC;
    __shared__ float sm_m[C::WARPS * C::LG], sm_s[C::WARPS * C::LG];
    __shared__ float sm_acc[C::WARPS * C::LG][HD];

    pdl_wait();                                      // partials come from the previous grid
    pdl_launch_dependents();

    const int h = blockIdx.x, s = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int grp = lane / C::TPS, dt = lane % C::TPS;
    const int P = a.n_splits;
    const size_t row = (size_t)s * a.n_head + h;
    const float2 *ml = a.ws_ml + row * P;
    const float *oc = a.ws_o + row * (size_t)P * HD + dt * V;

    // stream this lane group's splits: sp = stride * i + first
    const int first = warp * C::LG + grp, stride = C::WARPS * C::LG;
    float m = -INFINITY, S = 0.f, acc[V];
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] = 0.f;
    for (int base = first; base < P; base += stride * C::BATCH) {
        float2 mlv[C::BATCH];
        float ov[C::BATCH][V];
#pragma unroll
        for (int b = 0; b < C::BATCH; ++b) {
            const int sp = base + b * stride;
            mlv[b] = sp < P ? ml[sp] : make_float2(-INFINITY, 0.f);
            const float *src = oc + (size_t)(sp < P ? sp : 0) * HD;
#pragma unroll
            for (int i = 0; i < V; i += 4) {
                const float4 t = *reinterpret_cast<const float4 *>(src + i);
                ov[b][i] = t.x; ov[b][i + 1] = t.y; ov[b][i + 2] = t.z; ov[b][i + 3] = t.w;
            }
        }
#pragma unroll
        for (int b = 0; b < C::BATCH; ++b) fold<V>(m, S, acc, mlv[b].x, mlv[b].y, ov[b]);
    }
    // fold the lane groups and warps: publish, then thread d folds dim d
    const int slot = warp * C::LG + grp;
    if (dt == 0) {
        sm_m[slot] = m;
        sm_s[slot] = S;
    }
#pragma unroll
    for (int i = 0; i < V; ++i) sm_acc[slot][dt * V + i] = acc[i];
    __syncthreads();
    for (int d = threadIdx.x; d < HD; d += C::THREADS) {
        float M = -INFINITY, St = 0.f, A[1] = {0.f};
        for (int k = 0; k < C::WARPS * C::LG; ++k) {
            const float a2[1] = {sm_acc[k][d]};
            fold<1>(M, St, A, sm_m[k], sm_s[k], a2);
        }
        a.out[row * HD + d] = St > 0.f ? A[0] / St : 0.f;
    }
}

} // namespace attn
