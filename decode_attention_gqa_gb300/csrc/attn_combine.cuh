// attn_combine.cuh -- the combine kernel (step a7).
//
// minfer "10 · R4" §2.1/§3.2: per (sequence, query head), gmx = max over the
// splits of mx; each split is reweighted by w = exp(mx - gmx); S = sum w*S_sp,
// acc = sum w*oc_sp; o = acc / S, and 0 when S is 0 (every split empty).
//
// The same merge is evaluated as a fold so that every load of a block is in
// flight at once: a block covers one (sequence, head) and one 32-wide chunk
// of head_dim (more blocks than heads, so the partials stream through many
// SMs); each group of lanes folds its share of the splits into a running
// (m, S, acc) with the §2.1 update rule, a batch of splits at a time (the
// batch's maximum first, so that its weights are independent exponentials; a
// larger maximum rescales what came before; the batch is sized from the split
// count so that every load of a group leaves in one round where it can: each
// round is a dependent L2 round trip), the groups of a warp are folded
// with shuffles and the warps through shared memory. The result equals the
// two-pass form up to rounding.
// A split whose mx is -inf (no rows) is skipped, so an all-empty row gives
// o = 0 without evaluating -inf - (-inf). mx is in log2 units (the partial
// kernel folds log2 e into q), so the weights use the base-2 exponential.
#pragma once

#include "attn_device.cuh"

namespace attn {

template <int HD, int BATCH_ = 8>
struct CombineCfg {
    static constexpr int WARPS = 4;
    static constexpr int THREADS = WARPS * 32;
    static constexpr int DC = HD < 32 ? HD : 32;      // head_dim chunk per block
    static constexpr int NCHUNK = HD / DC;
    static constexpr int LPS = DC / 4;                // lanes per split row (float4 each)
    static constexpr int SPW = 32 / LPS;              // split groups per warp
    static constexpr int NG = WARPS * SPW;            // split groups per block
    static constexpr int BATCH = BATCH_;              // split rows in flight per lane
};

template <int HD, int BATCH>
__global__ void __launch_bounds__(CombineCfg<HD, BATCH>::THREADS)
attn_combine(const CombineArgs a)
{
    using C = CombineCfg<HD, BATCH>;
    __shared__ float sm_m[C::WARPS], sm_s[C::WARPS];
    __shared__ float sm_acc[C::WARPS][C::DC];

    // Let the next kernel's blocks get resident now (they wait for this grid
    // before touching anything it writes); the partials come from the grid
    // before this one.
    pdl_launch_dependents();
    pdl_wait();

    const int h = blockIdx.x, s = blockIdx.y, chunk = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sg = lane / C::LPS, dl = lane % C::LPS;
    const int P = a.n_splits;
    const size_t row = (size_t)s * a.n_head + h;
    const float2 *ml = a.ws_ml + row * P;
    const float *oc = a.ws_o + row * (size_t)P * HD + chunk * C::DC + dl * 4;

    // this lane group's splits: sp = group + NG * i
    const int group = warp * C::SPW + sg;
    float m = -INFINITY, S = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int base = group; base < P; base += C::NG * C::BATCH) {
        float2 mlv[C::BATCH];
        float ov[C::BATCH][4];
#pragma unroll
        for (int b = 0; b < C::BATCH; ++b) {
            const int sp = base + b * C::NG;
            float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
            mlv[b] = make_float2(-INFINITY, 0.f);
            if (sp < P) {                                     // past the last split: no load
                mlv[b] = ld_dep(ml + sp);
                t = ld_dep(reinterpret_cast<const float4 *>(oc + (size_t)sp * HD));
            }
            ov[b][0] = t.x; ov[b][1] = t.y; ov[b][2] = t.z; ov[b][3] = t.w;
        }
        // the batch's maximum first, then independent weights (no serial exp chain)
        float mb = m;
#pragma unroll
        for (int b = 0; b < C::BATCH; ++b) mb = fmaxf(mb, mlv[b].x);
        if (mb == -INFINITY) continue;                       // every split so far empty
        const float c0 = m == -INFINITY ? 0.f : ex2(m - mb);
        S *= c0;
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i] *= c0;
#pragma unroll
        for (int b = 0; b < C::BATCH; ++b) {
            // an empty split's o row was never written: skip it, never scale it by 0
            if (mlv[b].x == -INFINITY) continue;
            const float w = ex2(mlv[b].x - mb);
            S = fmaf(w, mlv[b].y, S);
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[i] = fmaf(w, ov[b][i], acc[i]);
        }
        m = mb;
    }
    // Fold the warp's split groups (lanes LPS apart hold the same dims) and
    // then the warps, each as maximum first, then one rescale and a sum, so
    // that the exponentials do not form a serial chain.
    float mw = m;
#pragma unroll
    for (int off = C::LPS; off < 32; off <<= 1) mw = fmaxf(mw, __shfl_xor_sync(0xffffffffu, mw, off));
    {
        const float c = m == -INFINITY ? 0.f : ex2(m - mw);   // a group that saw no split adds 0
        S *= c;
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i] *= c;
    }
#pragma unroll
    for (int off = C::LPS; off < 32; off <<= 1) {
        S += __shfl_xor_sync(0xffffffffu, S, off);
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], off);
    }
    if (sg == 0) {
        if (dl == 0) {
            sm_m[warp] = mw;
            sm_s[warp] = S;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) sm_acc[warp][dl * 4 + i] = acc[i];
    }
    __syncthreads();
    // the warps: thread d of the chunk
    if (threadIdx.x < C::DC) {
        const int d = threadIdx.x;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < C::WARPS; ++w) M = fmaxf(M, sm_m[w]);
        float St = 0.f, A = 0.f;
#pragma unroll
        for (int w = 0; w < C::WARPS; ++w) {
            const float wt = sm_m[w] == -INFINITY ? 0.f : ex2(sm_m[w] - M);
            St = fmaf(wt, sm_s[w], St);
            A = fmaf(wt, sm_acc[w][d], A);
        }
        a.out[row * HD + chunk * C::DC + d] = St > 0.f ? A / St : 0.f;
    }
}

} // namespace attn
