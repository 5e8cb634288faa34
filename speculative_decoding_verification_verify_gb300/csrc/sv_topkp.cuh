// sv_topkp.cuh -- per-row thresholds of top-k / top-p on the target distribution.
//
// p is the target distribution after temperature, top-k and top-p ("投机解码", section
// 接受规则为什么不改变分布: p already carries temperature, top-k and top-p).  Top-k keeps every token
// whose logit reaches the k-th largest logit; top-p then keeps the fewest whole value levels from
// the top whose probability, renormalised over the top-k set, reaches top_p.  Both keep a set
// {logit >= tau}, so one logit threshold per row describes the filter: the streaming fold, the
// finaliser, the rescan and the residual kernel treat logits below it as -inf.
//
// One CTA per row finds tau by radix descent over order-preserving keys of the logits (2 digit
// levels of 8 bits for bf16, 3 levels of 11, 11 and 10 bits for fp32): at each level a pass over
// the row histograms the next digit of the keys that match the chosen prefix (counts for top-k,
// masses 2^((l - max) * cs) for top-p) in shared memory, and one warp walks the bins from the top.
#pragma once

#include "sv_device.cuh"

namespace sv {

constexpr int NT_TK = 512;
constexpr int TK_BINS = 2048;

template <typename T>
struct KeyOf;

template <>
struct KeyOf<__nv_bfloat16> {
    static constexpr int LEVELS = 2;
    static __device__ __forceinline__ int shift(int lvl) { return lvl == 0 ? 8 : 0; }
    static __device__ __forceinline__ int bits(int) { return 8; }
    static __device__ __forceinline__ uint32_t key(const void *row, int64_t c)
    {
        const uint32_t u = __ldg((const unsigned short *)row + c);
        return (u & 0x8000u) ? (~u & 0xffffu) : (u | 0x8000u);
    }
    static __device__ __forceinline__ float value(uint32_t k)
    {
        const uint32_t u = (k & 0x8000u) ? (k & 0x7fffu) : (~k & 0xffffu);
        return __uint_as_float(u << 16);
    }
};

template <>
struct KeyOf<float> {
    static constexpr int LEVELS = 3;
    static __device__ __forceinline__ int shift(int lvl) { return lvl == 0 ? 21 : lvl == 1 ? 10 : 0; }
    static __device__ __forceinline__ int bits(int lvl) { return lvl == 2 ? 10 : 11; }
    static __device__ __forceinline__ uint32_t key(const void *row, int64_t c)
    {
        const uint32_t u = __float_as_uint(__ldg((const float *)row + c));
        return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    }
    static __device__ __forceinline__ float value(uint32_t k)
    {
        const uint32_t u = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
        return __uint_as_float(u);
    }
};

struct TopkpSmem {
    int cnt[TK_BINS];
    float mass[TK_BINS];
    float wmax[NT_TK / 32];
    int sel;          // chosen digit
    int above_cnt;    // count in bins above it
    float above_mass; // mass in bins above it
};

// One warp: the bins [0, nb) from the top; the first bin where the running count reaches `rank`
// (by_mass false) or the running mass reaches `target` (by_mass true).  Sets S.sel and the
// totals above it; when nothing reaches (rounding), the lowest non-empty bin.
__device__ __forceinline__ void walk_bins(TopkpSmem &S, int nb, bool by_mass, int rank, float target, int lane)
{
    const int per = nb / 32;  // nb is 256, 1024 or 2048
    // Lane l takes bins [nb - (l + 1) * per, nb - l * per), the top bins first.
    const int hi = nb - lane * per;
    float m = 0.f;
    int c = 0;
    for (int i = hi - 1; i >= hi - per; --i) {
        m += S.mass[i];
        c += S.cnt[i];
    }
    const bool ne = by_mass ? m > 0.f : c > 0;
    float mi = m;
    int ci = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float ym = __shfl_up_sync(0xffffffffu, mi, o);
        const int yc = __shfl_up_sync(0xffffffffu, ci, o);
        if (lane >= o) {
            mi += ym;
            ci += yc;
        }
    }
    const bool reach = ne && (by_mass ? mi >= target : ci >= rank);
    const unsigned hit = __ballot_sync(0xffffffffu, reach);
    const unsigned nonempty = __ballot_sync(0xffffffffu, ne);
    const int who = hit ? __ffs(hit) - 1 : (nonempty ? 31 - __clz(nonempty) : 31);
    if (lane == who) {
        float am = mi - m;
        int ac = ci - c;
        int sel = -1, lastne = hi - per;
        float lm = am;
        int lc = ac;
        for (int i = hi - 1; i >= hi - per; --i) {
            const bool bne = by_mass ? S.mass[i] > 0.f : S.cnt[i] > 0;
            if (bne) {
                if (hit && (by_mass ? am + S.mass[i] >= target : ac + S.cnt[i] >= rank)) {
                    sel = i;
                    break;
                }
                lastne = i;
                lm = am;
                lc = ac;
            }
            am += S.mass[i];
            ac += S.cnt[i];
        }
        S.sel = sel >= 0 ? sel : lastne;
        S.above_mass = sel >= 0 ? am : lm;
        S.above_cnt = sel >= 0 ? ac : lc;
    }
}

// Histogram of the next digit of the keys that match `prefix` on the bits above this level's
// digit and are >= floor_key: counts (MASS false) or masses 2^((l - mx) * cs) (MASS true).  The
// lanes of a warp that share a digit add their share once, through their lowest lane.
template <typename T, bool MASS>
__device__ void key_histogram(const void *row, int64_t V, uint32_t prefix, int lvl, uint32_t floor_key, float mx,
                              float cs, TopkpSmem &S)
{
    const int sh = KeyOf<T>::shift(lvl), nb = 1 << KeyOf<T>::bits(lvl);
    const int top = sh + KeyOf<T>::bits(lvl);
    const int lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < nb; i += NT_TK) {
        S.cnt[i] = 0;
        S.mass[i] = 0.f;
    }
    __syncthreads();
    for (int64_t base = 0; base < V; base += NT_TK) {
        const int64_t c = base + threadIdx.x;
        const uint32_t k = c < V ? KeyOf<T>::key(row, c) : 0u;
        const bool match = c < V && (top >= 32 || (k >> top) == (prefix >> top)) && k >= floor_key;
        const unsigned active = __ballot_sync(0xffffffffu, match);
        if (match) {
            const int d = (int)((k >> sh) & (uint32_t)(nb - 1));
            const unsigned grp = __match_any_sync(active, d);
            const int leader = __ffs(grp) - 1;
            if (MASS) {
                const float x = ex2((KeyOf<T>::value(k) - mx) * cs);
                float sum = 0.f;
                for (unsigned g = grp; g; g &= g - 1) sum += __shfl_sync(grp, x, __ffs(g) - 1);
                if (lane == leader) atomicAdd(&S.mass[d], sum);
            } else if (lane == leader) {
                atomicAdd(&S.cnt[d], __popc(grp));
            }
        }
    }
    __syncthreads();
}

// Sum over the row of the masses of keys >= floor_key.
template <typename T>
__device__ float mass_at_or_above(const void *row, int64_t V, uint32_t floor_key, float mx, float cs, TopkpSmem &S)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float z = 0.f;
    for (int64_t c = threadIdx.x; c < V; c += NT_TK) {
        const uint32_t k = KeyOf<T>::key(row, c);
        if (k >= floor_key) z += ex2((KeyOf<T>::value(k) - mx) * cs);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    __syncthreads();
    if (lane == 0) S.wmax[warp] = z;
    __syncthreads();
    float t = 0.f;
    for (int w = 0; w < NT_TK / 32; ++w) t += S.wmax[w];
    __syncthreads();
    return t;
}

// Grid: one CTA per row.  thr[r] = the row's logit threshold, or -inf when the row is not
// filtered (top-k off and top-p off, or a greedy request).
template <typename T>
__global__ void __launch_bounds__(NT_TK) sv_topkp_kernel(const Params P)
{
    __shared__ TopkpSmem S;
    const int64_t r = blockIdx.x;
    const int b = (int)(r / P.rpr);
    const int64_t V = P.V;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float Tb = P.temps ? __ldg(P.temps + b) : 1.f;
    const int kk = P.top_k ? __ldg(P.top_k + b) : 0;
    const float pp = P.top_p ? __ldg(P.top_p + b) : 1.f;
    const bool use_k = kk >= 1 && (int64_t)kk < V, use_p = pp < 1.f;
    if (Tb == 0.f || (!use_k && !use_p)) {
        if (tid == 0) P.thr[r] = NEG_INF;
        return;
    }
    const float cs = P.temps ? cs_of(Tb) : P.cs;
    const void *row = reinterpret_cast<const T *>(P.logits) + r * V;
    // The row's largest logit, the masses' reference.
    float mx = NEG_INF;
    for (int64_t c = tid; c < V; c += NT_TK) mx = fmax_nan(mx, KeyOf<T>::value(KeyOf<T>::key(row, c)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmax_nan(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) S.wmax[warp] = mx;
    __syncthreads();
    mx = S.wmax[0];
    for (int w = 1; w < NT_TK / 32; ++w) mx = fmax_nan(mx, S.wmax[w]);
    __syncthreads();
    if (!(mx > NEG_INF) || mx != mx || mx == POS_INF) {  // the streaming pass flags such rows
        if (tid == 0) P.thr[r] = NEG_INF;
        return;
    }
    constexpr int LV = KeyOf<T>::LEVELS;
    // Top-k: the key of the k-th largest logit (counts only).
    uint32_t kkey = 0u;
    if (use_k) {
        int rank = kk;
        uint32_t prefix = 0u;
        for (int lvl = 0; lvl < LV; ++lvl) {
            key_histogram<T, false>(row, V, prefix, lvl, 0u, mx, cs, S);
            if (warp == 0) walk_bins(S, 1 << KeyOf<T>::bits(lvl), false, rank, 0.f, lane);
            __syncthreads();
            prefix |= (uint32_t)S.sel << KeyOf<T>::shift(lvl);
            rank -= S.above_cnt;
            __syncthreads();
        }
        kkey = prefix;
    }
    uint32_t pkey = kkey;
    if (use_p) {
        // Top-p within the top-k set: the fewest value levels from the top holding top_p of its mass.
        float target = pp * mass_at_or_above<T>(row, V, kkey, mx, cs, S);
        uint32_t prefix = 0u;
        for (int lvl = 0; lvl < LV; ++lvl) {
            key_histogram<T, true>(row, V, prefix, lvl, kkey, mx, cs, S);
            if (warp == 0) walk_bins(S, 1 << KeyOf<T>::bits(lvl), true, 0, target, lane);
            __syncthreads();
            prefix |= (uint32_t)S.sel << KeyOf<T>::shift(lvl);
            target -= S.above_mass;
            __syncthreads();
        }
        pkey = prefix > kkey ? prefix : kkey;
    }
    if (tid == 0) P.thr[r] = KeyOf<T>::value(pkey);
}

}  // namespace sv
