// sv_stream.cuh -- the streaming fold: each warp walks its contiguous segment of a logit row with
// 16-byte non-allocating loads (the next step's loads issued before the current step is folded)
// and folds every element into a running (max, sum of 2^(l*cs - mc)) or a running argmax.
#pragma once

#include <climits>

#include "sv_device.cuh"

namespace sv {

#ifndef SV_VPL
#define SV_VPL 4
#endif
constexpr int VPL = SV_VPL;            // 16-byte vectors per lane per step
constexpr int STEP_VEC = 32 * VPL;     // vectors per warp step

// ---------------------------------------------------------------------------------------------
// Packed fp32 pairs (sm_100+ f32x2 arithmetic): half the FMA-pipe instructions per element.
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ uint64_t f2(float lo, float hi)
{
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
    return d;
}

__device__ __forceinline__ float2 f2_split(uint64_t d)
{
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(d));
    return make_float2(lo, hi);
}

__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// ---------------------------------------------------------------------------------------------
// Accumulators.
// ---------------------------------------------------------------------------------------------
struct SampleAcc {
    float m = NEG_INF;                 // running max logit of the lane
    float mc = REF_NONE;               // m * cs once a finite logit was seen: the sums' reference
    uint64_t acc[4] = {0, 0, 0, 0};    // four fp32 pairs of partial sums of 2^(l*cs - mc)
    __device__ __forceinline__ float total() const
    {
        const float2 a = f2_split(f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3])));
        return a.x + a.y;
    }
};

struct GreedyAcc {
    float best = NEG_INF;
    int idx = INT_MAX;
};

// The lane's next child-token column (tokens whose mass is kept out of the sums and whose
// logits are captured instead).  A lane visits its columns in ascending order.
struct ExCursor {
    const int *col;
    const int *node;
    int cnt, ptr, next;
    float *caps;
    __device__ __forceinline__ void init(const int *c, const int *nd, int n, float *cp)
    {
        col = c;
        node = nd;
        cnt = n;
        ptr = 0;
        caps = cp;
        next = n > 0 ? c[0] : INT_MAX;
    }
    __device__ __forceinline__ void advance()
    {
        ++ptr;
        next = ptr < cnt ? col[ptr] : INT_MAX;
    }
};

__device__ __forceinline__ void sample_rescale(SampleAcc &a, float vmax, float cs)
{
    if (vmax > a.m) {
        const float mcn = vmax * cs;
        const float f = ex2(a.mc - mcn);
        const uint64_t ff = f2(f, f);
#pragma unroll
        for (int j = 0; j < 4; ++j) a.acc[j] = f2_mul(a.acc[j], ff);
        a.m = vmax;
        a.mc = mcn;
    }
}

template <typename T>
__device__ __forceinline__ uint4 neg_inf_vec()
{
    const uint32_t n = sizeof(T) == 2 ? 0xFF80FF80u : 0xFF800000u;
    return make_uint4(n, n, n, n);
}

// Fold one 16-byte vector at column col into the sums; child tokens are zeroed and captured.
template <typename T>
__device__ __forceinline__ void sample_vec(SampleAcc &a, const uint4 &w, int col, float cs,
                                           uint64_t cs2, uint64_t nmc2, ExCursor &ex)
{
    constexpr int VEC = Elt<T>::VEC;
    constexpr int NP = VEC / 2;
    uint64_t e[NP];
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int p = 0; p < NP; ++p) {
        uint64_t x2;
        if (VEC == 8) x2 = f2(bf_lo(ww[p]), bf_hi(ww[p]));
        else x2 = f2(__uint_as_float(ww[2 * p]), __uint_as_float(ww[2 * p + 1]));
        const float2 z = f2_split(f2_fma(x2, cs2, nmc2));
        e[p] = f2(ex2(z.x), ex2(z.y));
    }
    if (col + VEC > ex.next) {
        // Rare: a child token lies in this vector (or was passed by this lane).
        float x[VEC], s[VEC];
        Elt<T>::unpack(w, x);
#pragma unroll
        for (int j = 0; j < VEC; ++j) s[j] = ex2(fmaf(x[j], cs, -a.mc));
        while (ex.next < col + VEC) {
            if (ex.next >= col) {
                float xv = 0.f;
#pragma unroll
                for (int j = 0; j < VEC; ++j) {
                    if (col + j == ex.next) {
                        s[j] = 0.f;
                        xv = x[j];
                    }
                }
                ex.caps[ex.node[ex.ptr]] = xv;
            }
            ex.advance();
        }
#pragma unroll
        for (int p = 0; p < NP; ++p) e[p] = f2(s[2 * p], s[2 * p + 1]);
    }
#pragma unroll
    for (int p = 0; p < NP; ++p) a.acc[p & 3] = f2_add(a.acc[p & 3], e[p]);
}

__device__ __forceinline__ void sample_scalar(SampleAcc &a, float x, int col, float cs, ExCursor &ex)
{
    sample_rescale(a, x, cs);
    float e = ex2(fmaf(x, cs, -a.mc));
    while (ex.next <= col) {
        if (ex.next == col) {
            e = 0.f;
            ex.caps[ex.node[ex.ptr]] = x;
        }
        ex.advance();
    }
    a.acc[0] = f2_add(a.acc[0], f2(e, 0.f));
}

__device__ __forceinline__ void greedy_scalar(GreedyAcc &a, float x, int col)
{
    if (x != x) {
        if (a.best == a.best) {
            a.best = x;
            a.idx = col;
        }
    } else if (x > a.best) {
        a.best = x;
        a.idx = col;
    }
}

// Max of the step's vectors (NaN if any element is NaN).
template <typename T>
__device__ __forceinline__ float step_max(const uint4 (&w)[VPL])
{
    if (sizeof(T) == 2) {
        uint32_t m = bmax2_nan(bmax2_nan(w[0].x, w[0].y), bmax2_nan(w[0].z, w[0].w));
#pragma unroll
        for (int u = 1; u < VPL; ++u)
            m = bmax2_nan(m, bmax2_nan(bmax2_nan(w[u].x, w[u].y), bmax2_nan(w[u].z, w[u].w)));
        return fmax_nan(bf_lo(m), bf_hi(m));
    } else {
        float m = Elt<float>::vmax(w[0]);
#pragma unroll
        for (int u = 1; u < VPL; ++u) m = fmax_nan(m, Elt<float>::vmax(w[u]));
        return m;
    }
}

// Greedy: on a new step maximum, locate its first occurrence (the lane's vectors in column order).
template <typename T>
__device__ __forceinline__ void greedy_step(GreedyAcc &a, const uint4 (&w)[VPL], int col0, float vmax)
{
    constexpr int VEC = Elt<T>::VEC;
    if (!(vmax > a.best) && vmax == vmax) return;
    if (vmax != vmax) {
        if (a.best == a.best) {
            a.best = vmax;
            a.idx = col0;
        }
        return;
    }
    int found = INT_MAX;
#pragma unroll
    for (int u = VPL - 1; u >= 0; --u) {
        float x[VEC];
        Elt<T>::unpack(w[u], x);
#pragma unroll
        for (int j = VEC - 1; j >= 0; --j)
            if (x[j] == vmax) found = col0 + u * 32 * VEC + j;
    }
    a.best = vmax;
    a.idx = found;
}

// Fold one step (VPL vectors per lane at columns col0 + u*32*VEC; those at step index >= nv are
// fillers holding -inf, whose columns belong to the next warp's segment).
template <typename T, bool SAMPLE>
__device__ __forceinline__ void fold_step(const uint4 (&w)[VPL], int nv, int col0, int lane, float cs,
                                          uint64_t cs2, ExCursor &ex, SampleAcc &sa, GreedyAcc &ga)
{
    constexpr int VEC = Elt<T>::VEC;
    const float vmax = step_max<T>(w);
    if (SAMPLE) {
        sample_rescale(sa, vmax, cs);
        const float nmc = -sa.mc;
        const uint64_t nmc2 = f2(nmc, nmc);
#pragma unroll
        for (int u = 0; u < VPL; ++u)
            if (lane + 32 * u < nv) sample_vec<T>(sa, w[u], col0 + u * 32 * VEC, cs, cs2, nmc2, ex);
    } else {
        greedy_step<T>(ga, w, col0, vmax);
    }
}

// Stream the 16-byte aligned body [b0, b1) of a warp segment: two steps per lane in flight.
template <typename T, bool SAMPLE>
__device__ __forceinline__ void stream_body(const T *row, int b0, int b1, int lane, float cs,
                                            ExCursor &ex, SampleAcc &sa, GreedyAcc &ga)
{
    constexpr int VEC = Elt<T>::VEC;
    const int nvec = (b1 - b0) / VEC;
    if (nvec <= 0) return;
    const uint4 *vp = reinterpret_cast<const uint4 *>(row + b0);
    const int nst = (nvec + STEP_VEC - 1) / STEP_VEC;
    const uint64_t cs2 = f2(cs, cs);
    uint4 cur[VPL], nxt[VPL];
#pragma unroll
    for (int u = 0; u < VPL; ++u) {
        const int v = lane + 32 * u;
        cur[u] = v < nvec ? ldg_stream(vp + v) : neg_inf_vec<T>();
    }
    for (int s = 0; s < nst; ++s) {
        const int nb = (s + 1) * STEP_VEC + lane;
#pragma unroll
        for (int u = 0; u < VPL; ++u) {
            const int v = nb + 32 * u;
            nxt[u] = v < nvec ? ldg_stream(vp + v) : neg_inf_vec<T>();
        }
        const int nv = min(STEP_VEC, nvec - s * STEP_VEC);
        fold_step<T, SAMPLE>(cur, nv, b0 + (s * STEP_VEC + lane) * VEC, lane, cs, cs2, ex, sa, ga);
#pragma unroll
        for (int u = 0; u < VPL; ++u) cur[u] = nxt[u];
    }
}

}  // namespace sv
