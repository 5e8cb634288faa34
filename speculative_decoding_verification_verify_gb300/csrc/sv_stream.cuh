// sv_stream.cuh -- the streaming fold: a warp takes one chunk of a logit row at a time, loads it
// with 16-byte non-allocating loads (eight per lane per step), folds every element into a running
// (max, sum of 2^(l*cs - mc)) or a running argmax, and writes the chunk's record.
#pragma once

#include <climits>

#include "sv_device.cuh"

namespace sv {

#ifndef SV_VPL
#define SV_VPL 8
#endif
constexpr int VPL = SV_VPL;            // 16-byte vectors per lane per step
constexpr int STEP_VEC = 32 * VPL;     // vectors per warp step
static_assert(CHUNK_VEC % STEP_VEC == 0, "a chunk spans whole steps");

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

// The child tokens of the row being streamed (tokens whose mass is kept out of the sums and
// whose logits are captured instead): lane i stands for nodes i and i + 32 of the request, and
// col[h] is that node's token column when the node is a child of the row's node, else INT_MAX.
struct Kids {
    int col[2];
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

// Element j of a 16-byte vector, which is then replaced by -inf (so that it adds nothing to the
// sums and does not raise the running maximum).
template <typename T>
__device__ __forceinline__ float take_element(uint4 &w, int j)
{
    const int wi = sizeof(T) == 2 ? (j >> 1) : j;
    uint32_t word = wi == 0 ? w.x : wi == 1 ? w.y : wi == 2 ? w.z : w.w;
    float x;
    if (sizeof(T) == 2) {
        const bool hi = (j & 1) != 0;
        x = hi ? bf_hi(word) : bf_lo(word);
        word = hi ? ((word & 0x0000ffffu) | 0xff800000u) : ((word & 0xffff0000u) | 0x0000ff80u);
    } else {
        x = __uint_as_float(word);
        word = 0xff800000u;
    }
    if (wi == 0) w.x = word;
    else if (wi == 1) w.y = word;
    else if (wi == 2) w.z = word;
    else w.w = word;
    return x;
}

// Rare: child tokens lie in the step whose lane-0 vector starts at column lo (columns below hi
// hold loaded data; the filler vectors past the chunk's body are left alone).  Each is captured
// by the lane that holds it and masked out of its vector.
template <typename T>
__device__ __forceinline__ void exclude_step(uint4 (&w)[VPL], int lo, int hi, int lane, const Kids &kd,
                                          float *caps, int rpr)
{
    constexpr int VEC = Elt<T>::VEC;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        unsigned m = __ballot_sync(0xffffffffu, kd.col[h] >= lo && kd.col[h] < hi);
        while (m) {
            const int src = __ffs(m) - 1;
            m &= m - 1;
            const int c = __shfl_sync(0xffffffffu, kd.col[h], src);
            const int v = (c - lo) / VEC;
            if ((v & 31) == lane) {
                const int u = v >> 5, j = c - lo - v * VEC;
#pragma unroll
                for (int uu = 0; uu < VPL; ++uu)
                    if (uu == u) {
                        const float x = take_element<T>(w[uu], j);
                        if (SV_INB(src + 32 * h, rpr, 203)) caps[src + 32 * h] = x;
                    }
            }
        }
    }
}

// Whether column col (a head or tail element of this lane, when has) is a child token; if so its
// logit x is captured.
__device__ __forceinline__ bool scalar_is_child(int col, bool has, float x, int lo, int hi, int lane,
                                                const Kids &kd, float *caps, int rpr)
{
    bool child = false;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        unsigned m = __ballot_sync(0xffffffffu, kd.col[h] >= lo && kd.col[h] < hi);
        while (m) {
            const int src = __ffs(m) - 1;
            m &= m - 1;
            const int c = __shfl_sync(0xffffffffu, kd.col[h], src);
            if (has && c == col) {
                child = true;
                if (SV_INB(src + 32 * h, rpr, 204)) caps[src + 32 * h] = x;
            }
        }
    }
    return child;
}

// One element outside the vector body (a row's unaligned head or tail); with a top-k / top-p
// threshold, logits below it weigh 0 (the row's maximum is always kept, so the reference stays).
template <bool FILT>
__device__ __forceinline__ void sample_scalar(SampleAcc &a, float x, float cs, float thr)
{
    sample_rescale(a, x, cs);
    if (!FILT || x >= thr) a.acc[0] = f2_add(a.acc[0], f2(ex2(fmaf(x, cs, -a.mc)), 0.f));
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

// Fold a lane's step (child tokens already masked to -inf): no per-vector checks; filler and
// masked elements add 2^-inf = 0 to the sums.
template <typename T, bool FILT>
__device__ __forceinline__ void sample_step_fast(SampleAcc &a, const uint4 (&w)[VPL], uint64_t cs2,
                                                 uint64_t nmc2, float thr)
{
    constexpr int NP = Elt<T>::VEC / 2;
#pragma unroll
    for (int u = 0; u < VPL; ++u) {
        const uint32_t ww[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
#pragma unroll
        for (int p = 0; p < NP; ++p) {
            const float xlo = NP == 4 ? bf_lo(ww[p]) : __uint_as_float(ww[2 * p]);
            const float xhi = NP == 4 ? bf_hi(ww[p]) : __uint_as_float(ww[2 * p + 1]);
            const uint64_t x2 = f2(xlo, xhi);
            float2 z = f2_split(f2_fma(x2, cs2, nmc2));
            if (FILT) {  // below the row's top-k / top-p threshold: weight 0
                z.x = xlo >= thr ? z.x : NEG_INF;
                z.y = xhi >= thr ? z.y : NEG_INF;
            }
            const int j = (u * NP + p) & 3;
            a.acc[j] = f2_add(a.acc[j], f2(ex2(z.x), ex2(z.y)));
        }
    }
}

// Fold one step (VPL vectors per lane at columns lo + (lane + 32 * u) * VEC; columns from hi on
// are fillers holding -inf, which belong to the next chunk).
template <typename T, bool SAMPLE, bool FILT>
__device__ __forceinline__ void fold_step(uint4 (&w)[VPL], int lo, int hi, int lane, float cs, uint64_t cs2,
                                          const Kids &kd, float *caps, int rpr, SampleAcc &sa, GreedyAcc &ga,
                                          float thr)
{
    if (SAMPLE) {
        const bool mine = (kd.col[0] >= lo && kd.col[0] < hi) || (kd.col[1] >= lo && kd.col[1] < hi);
        if (__any_sync(0xffffffffu, mine)) exclude_step<T>(w, lo, hi, lane, kd, caps, rpr);
        const float smax = step_max<T>(w);
        sample_rescale(sa, smax, cs);
        // Filtered: a step in which no lane holds a logit at or above the row's threshold adds
        // only zeros (most steps of a row, whose top-k set is small), so its exponentials are
        // skipped; the sums are the same.
        if (FILT && !__any_sync(0xffffffffu, smax >= thr)) return;
        const float nmc = -sa.mc;
        sample_step_fast<T, FILT>(sa, w, cs2, f2(nmc, nmc), thr);
    } else {
        greedy_step<T>(ga, w, lo + lane * Elt<T>::VEC, step_max<T>(w));
    }
}

// Flush the warp's accumulators into record `idx` (lane 0 writes it) and restart the sums; a
// lane keeps its reference mc, so later records stay in the same scaled domain per lane.  A
// sampling record also carries the columns [c0, c1) it covers.
template <bool SAMPLE>
__device__ __forceinline__ void flush_record(float4 *rec, bool rec_ok, int lane, SampleAcc &sa, GreedyAcc &ga, int c0,
                                             int c1)
{
    float4 out;
    if (SAMPLE) {
        float mc = sa.mc, sum = sa.total();
        warp_rec_merge(mc, sum);
        out = make_float4(mc, sum, __int_as_float(c0), __int_as_float(c1));
#pragma unroll
        for (int j = 0; j < 4; ++j) sa.acc[j] = 0;
    } else {
        float v = ga.best;
        int i = ga.idx;
        warp_arg_merge(v, i);
        out = make_float4(v, __int_as_float(i), 0.f, 0.f);
        ga.best = NEG_INF;
        ga.idx = INT_MAX;
    }
    if (lane == 0 && rec_ok) *rec = out;
}

// One lane's loads of a step: vectors p[32*u]; with CHECK, those at 32*u >= lim are -inf fillers.
// el is p's first element in the flat logits array of `total` elements (checked in debug builds).
#ifndef SV_STREAM_EF
#define SV_STREAM_EF 1
#endif
// EF: evict-first loads (with SV_STREAM_EF; the filtered pass, whose rows the threshold pass read
// just before).
template <typename T, bool CHECK, bool EF = false>
__device__ __forceinline__ void load_step(uint4 (&d)[VPL], const uint4 *p, int lim, int64_t el, int64_t total)
{
    [[maybe_unused]] constexpr int VEC = Elt<T>::VEC;
#pragma unroll
    for (int u = 0; u < VPL; ++u)
        d[u] = ((!CHECK || 32 * u < lim) && SV_INB(el + (int64_t)(32 * u + 1) * VEC - 1, total, 201))
                   ? ((EF && SV_STREAM_EF) ? ldg_stream_ef(p + 32 * u) : ldg_stream(p + 32 * u))
                   : neg_inf_vec<T>();
}

// One warp streams chunk sg of a row: the body's first step and the head and tail elements are
// loaded first (the caller may update kd meanwhile through `ready`), then the steps are folded
// and the chunk's record is written to *rec (when rec_ok).  rowflat is the row's first element in
// the flat logits array of `total` elements, rpr the request's rows (both for the range checks of
// debug builds).
template <typename T, bool SAMPLE, bool FILT, typename Ready>
__device__ __forceinline__ void stream_chunk(const T *row, const Seg &sg, int lane, float cs, Kids &kd, float *caps,
                                             float4 *rec, Ready ready, float thr, int64_t rowflat, int64_t total,
                                             int rpr, bool rec_ok)
{
    constexpr int VEC = Elt<T>::VEC;
    const int c0 = (int)sg.c0, b0 = (int)sg.b0, b1 = (int)sg.b1, c1 = (int)sg.c1;
    const int nvec = (b1 - b0) / VEC;
    const uint4 *vp = reinterpret_cast<const uint4 *>(row + b0) + lane;
    const int64_t el = rowflat + b0 + (int64_t)lane * VEC;
    uint4 cur[VPL];
    if (nvec >= STEP_VEC) load_step<T, false, FILT>(cur, vp, 0, el, total);
    else if (nvec > 0) load_step<T, true, FILT>(cur, vp, nvec - lane, el, total);
    const bool has_head = c0 + lane < b0 && SV_INB(rowflat + c0 + lane, total, 202);
    const bool has_tail = b1 + lane < c1 && SV_INB(rowflat + b1 + lane, total, 202);
    const float xh = has_head ? Elt<T>::load(row, c0 + lane) : 0.f;
    const float xt = has_tail ? Elt<T>::load(row, b1 + lane) : 0.f;
    ready();
    SampleAcc sa;
    GreedyAcc ga;
    if (b0 > c0) {  // warp-uniform
        if (SAMPLE) {
            if (!scalar_is_child(c0 + lane, has_head, xh, c0, b0, lane, kd, caps, rpr) && has_head)
                sample_scalar<FILT>(sa, xh, cs, thr);
        } else if (has_head) {
            greedy_scalar(ga, xh, c0 + lane);
        }
    }
    const uint64_t cs2 = f2(cs, cs);
    const int nst = (nvec + STEP_VEC - 1) / STEP_VEC;
    for (int s = 0; s < nst; ++s) {
        if (s > 0) {
            const int64_t es = el + (int64_t)s * STEP_VEC * VEC;
            if (nvec - s * STEP_VEC >= STEP_VEC) load_step<T, false, FILT>(cur, vp + s * STEP_VEC, 0, es, total);
            else load_step<T, true, FILT>(cur, vp + s * STEP_VEC, nvec - s * STEP_VEC - lane, es, total);
        }
        const int lo = b0 + s * STEP_VEC * VEC;
        const int hi = min(lo + STEP_VEC * VEC, b1);
        fold_step<T, SAMPLE, FILT>(cur, lo, hi, lane, cs, cs2, kd, caps, rpr, sa, ga, thr);
    }
    if (c1 > b1) {  // warp-uniform
        if (SAMPLE) {
            if (!scalar_is_child(b1 + lane, has_tail, xt, b1, c1, lane, kd, caps, rpr) && has_tail)
                sample_scalar<FILT>(sa, xt, cs, thr);
        } else if (has_tail) {
            greedy_scalar(ga, xt, b1 + lane);
        }
    }
    flush_record<SAMPLE>(rec, rec_ok, lane, sa, ga, c0, c1);
}

// ---------------------------------------------------------------------------------------------
// The streaming warp's view of a request's nodes: lane i holds nodes i and i + 32 (token and
// parent; the chain is a path tree), and Kids marks the children of row n's node with a usable
// token.
// ---------------------------------------------------------------------------------------------
struct NodeView {
    int tok[2], par[2];
};

__device__ __forceinline__ void load_nodes(const Params &P, int b, int lane, NodeView &nv)
{
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int m = lane + 32 * h;
        nv.tok[h] = -1;
        nv.par[h] = -1;
        if (m >= 1 && m < P.rpr) {
            nv.tok[h] = node_token(P, b, m);
            nv.par[h] = node_parent(P, b, m);
        }
    }
}

__device__ __forceinline__ void kids_of(const Params &P, const NodeView &nv, int n, Kids &kd)
{
#pragma unroll
    for (int h = 0; h < 2; ++h)
        kd.col[h] = (nv.par[h] == n && nv.tok[h] >= 0 && (int64_t)nv.tok[h] < P.V) ? nv.tok[h] : INT_MAX;
}

}  // namespace sv
