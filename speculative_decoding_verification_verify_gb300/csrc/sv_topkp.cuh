// sv_topkp.cuh -- per-row thresholds of top-k / top-p on the target distribution.
//
// p is the target distribution after temperature, top-k and top-p ("投机解码", section
// 接受规则为什么不改变分布: p already carries temperature, top-k and top-p).  Top-k keeps every token
// whose logit reaches the k-th largest logit; top-p then keeps the fewest whole value levels from
// the top whose probability, renormalised over the top-k set, reaches top_p.  Both keep a set
// {logit >= tau}, so one logit threshold per row describes the filter: the streaming fold, the
// finaliser, the rescan and the residual kernel treat logits below it as -inf.
//
// One CTA per row finds tau by radix descent over order-preserving keys of the logits (8-bit
// digits: 2 levels for bf16, 4 for fp32): at each level a pass over the row (16-byte loads)
// histograms the next digit of the keys that match the chosen prefix (counts for top-k, masses
// 2^((l - max) * cs) for top-p) in per-warp shared-memory copies, and one warp walks the bins
// from the top.  The masses are fp32 terms summed in 64-bit fixed point (units of 2^-shift of the
// row maximum's term, shift = 62 - bits(V), so no row's sum overflows; integer atomics and exact
// sums, GB300 having few fp64 units), so a row's top-p crossing is placed within about 2e-7 of
// its mass: the terms' own error, the truncation adding less than V^2 2^-62 of the maximum's term
// (4e-9 at V = 128256, below 1e-6 up to V = 2^21).
#pragma once

#include <climits>

#include "sv_device.cuh"

namespace sv {

#ifndef SV_NT_TK
#define SV_NT_TK 512
#endif
constexpr int NT_TK = SV_NT_TK;
constexpr int TK_BINS = 256;        // 8-bit digits
constexpr int TK_WARPS = NT_TK / 32;
#ifndef SV_TK_UNROLL
#define SV_TK_UNROLL 2
#endif
#ifndef SV_TK_CTAS
#define SV_TK_CTAS 2
#endif
constexpr int TK_UNROLL = SV_TK_UNROLL;  // 16-byte loads a thread keeps in flight in a pass
// A threshold slot the ring kernel (sv_topkp_ring.cuh) leaves to the general one (a NaN no row's
// threshold can be).
constexpr uint32_t TK_PENDING = 0x7fc0beefu;
constexpr int TK_CTAS = SV_TK_CTAS;      // threshold CTAs per SM (each holds one row at a time)

template <typename T>
struct KeyOf;

template <>
struct KeyOf<__nv_bfloat16> {
    static constexpr int LEVELS = 2;
    static constexpr int VEC = 8;
    static __device__ __forceinline__ int shift(int lvl) { return 8 * (LEVELS - 1 - lvl); }
    static __device__ __forceinline__ uint32_t key_of_bits(uint32_t u)
    {
        return (u & 0x8000u) ? (~u & 0xffffu) : (u | 0x8000u);
    }
    static __device__ __forceinline__ uint32_t key(const void *row, int64_t c)
    {
        return key_of_bits(__ldg((const unsigned short *)row + c));
    }
    // The VEC keys of a 16-byte vector.
    static __device__ __forceinline__ void keys(const uint4 &w, uint32_t (&k)[VEC])
    {
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            k[2 * i] = key_of_bits(ww[i] & 0xffffu);
            k[2 * i + 1] = key_of_bits(ww[i] >> 16);
        }
    }
    static __device__ __forceinline__ float value(uint32_t k)
    {
        const uint32_t u = (k & 0x8000u) ? (k & 0x7fffu) : (~k & 0xffffu);
        return __uint_as_float(u << 16);
    }
};

template <>
struct KeyOf<float> {
    static constexpr int LEVELS = 4;
    static constexpr int VEC = 4;
    static __device__ __forceinline__ int shift(int lvl) { return 8 * (LEVELS - 1 - lvl); }
    static __device__ __forceinline__ uint32_t key_of_bits(uint32_t u)
    {
        return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    }
    static __device__ __forceinline__ uint32_t key(const void *row, int64_t c)
    {
        return key_of_bits(__float_as_uint(__ldg((const float *)row + c)));
    }
    static __device__ __forceinline__ void keys(const uint4 &w, uint32_t (&k)[VEC])
    {
        k[0] = key_of_bits(w.x);
        k[1] = key_of_bits(w.y);
        k[2] = key_of_bits(w.z);
        k[3] = key_of_bits(w.w);
    }
    static __device__ __forceinline__ float value(uint32_t k)
    {
        const uint32_t u = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
        return __uint_as_float(u);
    }
};

constexpr int TK_SPAN = 2048;  // keys the ring kernel's exact histogram covers below the row maximum

struct TopkpSmem {
    int cnt[TK_BINS];
    double mass[TK_BINS];
    union {                          // per-warp histograms of one pass, merged into cnt / mass
        int wcnt[TK_WARPS][TK_BINS];
        unsigned long long wmass[TK_WARPS][TK_BINS];  // fixed point (see fixed_term)
    };
    float wmax[NT_TK / 32];
    unsigned long long wz[TK_WARPS];  // per-warp sums of the fine top-p pass
    int sel;           // chosen digit (the fine top-p pass: the chosen key's distance from the maximum's)
    int above_cnt;     // count in bins above it
    double above_mass; // mass in bins above it
};

// One warp: the bins [0, nb) from the top; the first bin where the running count reaches `rank`
// (by_mass false) or the running mass reaches `target` (by_mass true).  Sets S.sel and the
// totals above it; when nothing reaches (rounding), the lowest non-empty bin.
__device__ __forceinline__ void walk_bins(TopkpSmem &S, int nb, bool by_mass, int rank, double target, int lane)
{
    const int per = nb / 32;  // nb is 256
    // Lane l takes bins [nb - (l + 1) * per, nb - l * per), the top bins first.
    const int hi = nb - lane * per;
    double m = 0.0;
    int c = 0;
    for (int i = hi - 1; i >= hi - per; --i) {
        m += S.mass[i];
        c += S.cnt[i];
    }
    const bool ne = by_mass ? m > 0.0 : c > 0;
    double mi = m;
    int ci = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double ym = __shfl_up_sync(0xffffffffu, mi, o);
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
        double am = mi - m;
        int ac = ci - c;
        int sel = -1, lastne = hi - per;
        double lm = am;
        int lc = ac;
        for (int i = hi - 1; i >= hi - per; --i) {
            const bool bne = by_mass ? S.mass[i] > 0.0 : S.cnt[i] > 0;
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

// Visit the keys of a row (row = column 0, rowflat its flat index, mis the logits base's
// misalignment in elements): the 16-byte aligned body with vector loads, UNR of them in flight a
// thread, the head and tail element by element.  f(key) is called for each element of the head
// and tail, g(keys) once for each visited vector of the body.  With MAX, vmx takes the largest
// logit of every element (NaN if one is NaN).  With SKIP, a vector whose largest logit is below
// fl (a value, not NaN) is not visited: none of its keys can reach the key of fl.
template <typename T, bool MAX, bool SKIP, int UNR, typename F, typename G>
__device__ __forceinline__ void for_each_vec(const void *row, int64_t rowflat, int64_t V, int mis, float fl,
                                             float &vmx, F f, G g)
{
    constexpr int VEC = KeyOf<T>::VEC;
    const int64_t a0 = min((int64_t)((VEC - (rowflat + mis) % VEC) % VEC), V);
    const int64_t nv = (V - a0) / VEC;
    const int64_t a1 = a0 + nv * VEC;
    auto one = [&](int64_t c) {
        const uint32_t k = KeyOf<T>::key(row, c);
        if (MAX) vmx = fmax_nan(vmx, KeyOf<T>::value(k));
        f(k);
    };
    for (int64_t c = threadIdx.x; c < a0; c += NT_TK) one(c);
    for (int64_t c = a1 + threadIdx.x; c < V; c += NT_TK) one(c);
    // UNR vectors per thread in flight: a pass is bound by the loads' latency otherwise.
    const uint4 *vp = reinterpret_cast<const uint4 *>(reinterpret_cast<const T *>(row) + a0);
    for (int64_t i0 = threadIdx.x; i0 < nv; i0 += (int64_t)UNR * NT_TK) {
        uint4 w[UNR];
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
            const int64_t i = i0 + (int64_t)u * NT_TK;
            if (i < nv) w[u] = ldg_stream(vp + i);
        }
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
            if (i0 + (int64_t)u * NT_TK >= nv) break;
            if (MAX || SKIP) {
                const float m = Elt<T>::vmax(w[u]);
                if (MAX) vmx = fmax_nan(vmx, m);
                if (SKIP && !(m >= fl)) continue;
            }
            uint32_t k[VEC];
            KeyOf<T>::keys(w[u], k);
            g(k);
        }
    }
}

// The same visit with f called for every element, TK_UNROLL vectors in flight.
template <typename T, bool MAX, bool SKIP, typename F>
__device__ __forceinline__ void for_each_key(const void *row, int64_t rowflat, int64_t V, int mis, float fl,
                                             float &vmx, F f)
{
    constexpr int VEC = KeyOf<T>::VEC;
    for_each_vec<T, MAX, SKIP, TK_UNROLL>(row, rowflat, V, mis, fl, vmx, f, [&](const uint32_t (&k)[VEC]) {
#pragma unroll
        for (int e = 0; e < VEC; ++e) f(k[e]);
    });
}

// A term t >= 0 as an integer in units of 2^-shift, rounded down (an error below 2^-shift), for
// t 2^shift < 2^62: the bit pattern's mantissa shifted by its exponent, integer operations only.
__device__ __forceinline__ unsigned long long fixed_term(float t, int shift)
{
    const uint32_t u = __float_as_uint(t);
    const int ex = (int)(u >> 23) - 127;  // t = 1.m * 2^ex
    if (!(t > 0.f) || ex + shift < 0) return 0ull;
    const unsigned long long m = (u & 0x7fffffu) | 0x800000u;
    const int s = ex + shift - 23;
    return s >= 0 ? m << s : m >> (-s);
}

// The fixed-point unit of a row of V terms in [0, 1]: V * 2^shift stays below 2^62.
__device__ __forceinline__ int mass_shift(int64_t V)
{
    return 62 - (64 - __clzll((long long)V));
}

// Histogram of the next digit of the keys that match `prefix` on the bits above this level's
// digit and are >= floor_key: counts (MASS false) or masses 2^((l - mx) * cs) (MASS true).  Each
// warp adds every counted key to its own copy with a shared-memory atomic, and the copies are
// merged at the end.  (Adding a thread's runs of equal digits at once was slower: consecutive
// logits rarely share a digit, and the run test makes the warp diverge.)  Every counted key is at least
// max(prefix, floor_key) (prefix has zeros below this level's digit), so vectors whose largest
// logit lies below that key's value are skipped whole.  MAX (first level only): *mx_out = the
// row's largest logit as seen by this thread, NaN if it saw a NaN.
template <typename T, bool MASS, bool MAX = false>
__device__ void key_histogram(const void *row, int64_t rowflat, int64_t V, int mis, uint32_t prefix, int lvl,
                              uint32_t floor_key, float mx, float cs, TopkpSmem &S, float *mx_out = nullptr)
{
    const int sh = KeyOf<T>::shift(lvl);
    const int top = sh + 8;
    const int warp = threadIdx.x >> 5;
    if (MASS)
        for (int i = threadIdx.x; i < TK_WARPS * TK_BINS; i += NT_TK) (&S.wmass[0][0])[i] = 0ull;
    else
        for (int i = threadIdx.x; i < TK_WARPS * TK_BINS; i += NT_TK) (&S.wcnt[0][0])[i] = 0;
    __syncthreads();
    // The skip bound: the value of the smallest key that can be counted, when it lies above the
    // key of -inf (a NaN-free row's keys lie between those of -inf and +inf).
    const uint32_t fk = prefix > floor_key ? prefix : floor_key;
    const float fl = KeyOf<T>::value(fk);
    const bool skip = fk > KeyOf<T>::key_of_bits(sizeof(T) == 2 ? 0xff80u : 0xff800000u) && fl == fl;
    float vmx = NEG_INF;
    const int fsh = mass_shift(V);
    auto visit = [&](uint32_t k) {
        if ((top >= 32 || (k >> top) == (prefix >> top)) && k >= floor_key) {
            const int d = (int)((k >> sh) & 0xffu);
            if (MASS) atomicAdd(&S.wmass[warp][d], fixed_term(ex2((KeyOf<T>::value(k) - mx) * cs), fsh));
            else atomicAdd(&S.wcnt[warp][d], 1);
        }
    };
    if (!MAX && skip) for_each_key<T, false, true>(row, rowflat, V, mis, fl, vmx, visit);
    else for_each_key<T, MAX, false>(row, rowflat, V, mis, fl, vmx, visit);
    if (MAX) *mx_out = vmx;
    __syncthreads();
    for (int i = threadIdx.x; i < TK_BINS; i += NT_TK) {
        int c = 0;
        unsigned long long m = 0ull;
        if (MASS)
            for (int w = 0; w < TK_WARPS; ++w) m += S.wmass[w][i];
        else
            for (int w = 0; w < TK_WARPS; ++w) c += S.wcnt[w][i];
        S.cnt[i] = c;
        S.mass[i] = MASS ? ldexp((double)m, -fsh) : 0.0;  // 256 conversions a pass, not one per logit
    }
    __syncthreads();
}

// Keys of a 16-bit row the fine top-p pass can cover: one 64-bit mass bin each, in the space of
// the per-warp histograms.
constexpr int TK_FINE = TK_WARPS * TK_BINS;

// Top-p over the keys >= kkey of a row of 16-bit logits, in one histogram at full key resolution.
// Z = the set's mass in fixed point: zin when the caller's first pass summed it (top-p alone),
// else summed here.  Every key below
// x0 = mx + log2(Z (1 - p) / (2 V)) / cs weighs at most 2^((x0 - mx) cs), so all of them together
// hold at most half of the (1 - p) Z that lies outside the top-p set: the threshold is at least
// x0, and the walk from the top over the keys in [x0, mx] reaches p Z exactly where the walk over
// the whole row would.  One count per key there (32-bit shared-memory atomics spread over up to
// TK_FINE keys, where the top digit's 256 bins put a flat row's logits in a handful; a key's mass
// is its count times its term); false, with the shared state free for the digit passes, when
// that span is wider than TK_FINE.  pkey: the key of the threshold.
template <typename T>
__device__ __noinline__ bool topp_fine(const void *row, int64_t rowflat, int64_t V, int mis, uint32_t kkey, float mx, float cs,
                          float pp, unsigned long long zin, TopkpSmem &S, uint32_t &pkey)
{
    static_assert(sizeof(T) == 2, "16-bit keys");
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int fsh = mass_shift(V);
    const uint32_t ninf_key = KeyOf<T>::key_of_bits(0xff80u);
    float vmx = NEG_INF;
    constexpr int VEC = KeyOf<T>::VEC;
    constexpr int UNR = 4;  // vectors in flight a thread: these passes carry little state
    auto term = [&](uint32_t k) { return ex2((KeyOf<T>::value(k) - mx) * cs); };
    // Z over the set (keys >= kkey; vectors below kkey's value skipped when kkey lies above -inf):
    // a vector's terms summed in fp32, then added in fixed point (an error below 2^-45 a vector).
    unsigned long long z = 0ull;
    auto z1 = [&](uint32_t k) {
        if (k >= kkey) z += fixed_term(term(k), fsh);
    };
    auto zv = [&](const uint32_t (&k)[VEC]) {
        float t = 0.f;
#pragma unroll
        for (int e = 0; e < VEC; ++e) t += k[e] >= kkey ? term(k[e]) : 0.f;
        z += fixed_term(t, fsh);
    };
    unsigned long long Z = zin;
    if (Z == 0ull) {  // not summed by the caller's first pass
        if (kkey > ninf_key) for_each_vec<T, false, true, UNR>(row, rowflat, V, mis, KeyOf<T>::value(kkey), vmx, z1, zv);
        else for_each_vec<T, false, false, UNR>(row, rowflat, V, mis, 0.f, vmx, z1, zv);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
        if (lane == 0) S.wz[warp] = z;
        __syncthreads();
        for (int w = 0; w < TK_WARPS; ++w) Z += S.wz[w];
    }
    // The floor: x0's key rounded down, within [kkey, the maximum's key].
    const uint32_t mxkey = KeyOf<T>::key_of_bits(__float_as_uint(mx) >> 16);
    const float lg = log2f((float)Z) - (float)fsh + log2f(0.5f * (1.f - pp)) - log2f((float)V);
    const float x0 = mx + lg / cs;
    uint32_t fk = ninf_key;
    if (x0 > NEG_INF) {
        fk = KeyOf<T>::key_of_bits(__float_as_uint(x0) >> 16);  // the low bits cut: toward zero
        if (KeyOf<T>::value(fk) > x0) --fk;
    }
    fk = min(max(fk, kkey), mxkey);
    const int span = (int)(mxkey - fk) + 1;
    if (span > TK_FINE) {
        __syncthreads();  // S.wz read by every thread before the digit passes reuse S
        return false;
    }
    // One count per key of [fk, mxkey], bin 0 the maximum's; a key's mass is its count times its
    // term, formed once a bin in the walk.
    int *cnt = &S.wcnt[0][0];
    for (int i = tid; i < span; i += NT_TK) cnt[i] = 0;
    if (tid == 0) S.sel = 0x7fffffff;
    __syncthreads();
    auto h1 = [&](uint32_t k) {
        if (k >= fk && k <= mxkey) atomicAdd(&cnt[mxkey - k], 1);
    };
    auto hv = [&](const uint32_t (&k)[VEC]) {
#pragma unroll
        for (int e = 0; e < VEC; ++e) h1(k[e]);
    };
    if (fk > ninf_key) for_each_vec<T, false, true, UNR>(row, rowflat, V, mis, KeyOf<T>::value(fk), vmx, h1, hv);
    else for_each_vec<T, false, false, UNR>(row, rowflat, V, mis, 0.f, vmx, h1, hv);
    __syncthreads();
    // The walk: the first key from the top whose bin is not empty and whose running mass reaches
    // ceil(p Z).  Thread t holds bins [8t, 8t + 8); an exclusive block scan of their sums.
    constexpr int PT = TK_FINE / NT_TK;
    const double tgt = (double)pp * (double)Z;  // one fp64 product a row
    const unsigned long long target = tgt <= 0.0 ? 0ull : (unsigned long long)ceil(tgt);
    unsigned long long bm[PT];
    unsigned long long own = 0ull;
#pragma unroll
    for (int e = 0; e < PT; ++e) {
        const int i = PT * tid + e;
        const int c = i < span ? cnt[i] : 0;
        bm[e] = c > 0 ? (unsigned long long)c * fixed_term(term(mxkey - (uint32_t)i), fsh) : 0ull;
        own += bm[e];
    }
    unsigned long long incl = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    __syncthreads();  // every thread has read S.wz above
    if (lane == 31) S.wz[warp] = incl;
    __syncthreads();
    unsigned long long run = incl - own;
    for (int w = 0; w < warp; ++w) run += S.wz[w];
#pragma unroll
    for (int e = 0; e < PT; ++e) {
        run += bm[e];
        if (bm[e] > 0ull && run >= target) {
            atomicMin(&S.sel, PT * tid + e);
            break;
        }
    }
    __syncthreads();
    const int sel = S.sel;
    __syncthreads();  // S.sel read before the caller's next use of S
    // Not reached: only for a top-p within about 2e-7 of 1, where the fused first pass's Z (about
    // 1e-7 relative) can exceed the keys' exact total by more than the bound's margin; the digit
    // passes decide.
    if (sel == 0x7fffffff) return false;
    pkey = mxkey - (uint32_t)sel;
    return true;
}

// The threshold of row r: thr[r] = the row's logit threshold, or -inf when the row is not
// filtered (top-k off and top-p off, or a greedy request).
template <typename T>
__device__ void topkp_row(const Params &P, int64_t r, TopkpSmem &S)
{
    const int b = (int)(r / P.rpr);
    const int64_t V = P.V;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // The row, its request's options and its threshold slot (range-checked in debug builds).
    if (!(SV_INB(b, P.B, 701) && SV_INB(r, (int64_t)P.B * P.rpr, 702) && SV_INB(r * V + V - 1, P.total, 703))) return;
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
    const int64_t rowflat = r * V;
    constexpr int LV = KeyOf<T>::LEVELS;
    // First pass: the row's largest logit (the masses' reference; NaN if the row holds one) and
    // the top digit's counts, which top-k needs first.
    float mx = NEG_INF;
    // Top-p alone: the maximum, and for 16-bit logits the row's mass in the same read, summed
    // against this thread's running maximum mrun (rescaled when it grows; each vector's terms
    // summed in fp32, the vector sums added with compensation), so the fine pass needs no pass of
    // its own for Z (relative error about 1e-7, far inside the 1e-6 at which top-p boundaries are
    // told apart).
    constexpr bool FUSE = sizeof(T) == 2;
    float zrun = 0.f, zc = 0.f, mrun = NEG_INF;
    auto zadd = [&](float t) {
        const float y = t - zc, u = zrun + y;
        zc = (u - zrun) - y;
        zrun = u;
    };
    auto rebase = [&]() {  // mx: this thread's maximum so far, this vector's included
        if (mx > mrun) {
            const float f = mrun > NEG_INF ? ex2((mrun - mx) * cs) : 0.f;
            zrun *= f;
            zc *= f;
            mrun = mx;
        }
    };
    if (use_k) {
        key_histogram<T, false, true>(row, rowflat, V, P.mis, 0u, 0, 0u, 0.f, cs, S, &mx);
    } else if (FUSE && use_p) {
        for_each_vec<T, true, false, 4>(
            row, rowflat, V, P.mis, 0.f, mx,
            [&](uint32_t k) {
                rebase();
                if (mrun > NEG_INF) zadd(ex2((KeyOf<T>::value(k) - mrun) * cs));
            },
            [&](const uint32_t (&k)[KeyOf<T>::VEC]) {
                rebase();
                if (mrun > NEG_INF) {
                    float t = 0.f;
#pragma unroll
                    for (int e = 0; e < KeyOf<T>::VEC; ++e) t += ex2((KeyOf<T>::value(k[e]) - mrun) * cs);
                    zadd(t);
                }
            });
    } else {
        for_each_vec<T, true, false, 4>(row, rowflat, V, P.mis, 0.f, mx, [](uint32_t) {},  // the maximum only
                                        [](const uint32_t (&)[KeyOf<T>::VEC]) {});
    }
    const float mine = mx;  // this thread's maximum (mrun, when the mass was summed)
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
    // The fused pass's Z in fixed point: each thread's sum moved to the row maximum.
    unsigned long long zpre = 0ull;
    if (FUSE && !use_k && use_p) {
        const float zt = mine > NEG_INF ? (zrun - zc) * ex2((mine - mx) * cs) : 0.f;
        unsigned long long z = fixed_term(zt, mass_shift(V));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
        if (lane == 0) S.wz[warp] = z;
        __syncthreads();
        for (int w = 0; w < TK_WARPS; ++w) zpre += S.wz[w];
        __syncthreads();
    }
    // Top-k: the key of the k-th largest logit (counts only; the top digit's are in S already).
    uint32_t kkey = 0u;
    if (use_k) {
        int rank = kk;
        uint32_t prefix = 0u;
        for (int lvl = 0; lvl < LV; ++lvl) {
            if (lvl > 0) key_histogram<T, false>(row, rowflat, V, P.mis, prefix, lvl, 0u, mx, cs, S);
            if (warp == 0) walk_bins(S, TK_BINS, false, rank, 0.0, lane);
            __syncthreads();
            prefix |= (uint32_t)S.sel << KeyOf<T>::shift(lvl);
            rank -= S.above_cnt;
            __syncthreads();
        }
        kkey = prefix;
    }
    uint32_t pkey = kkey;
    bool fine = false;
    if constexpr (sizeof(T) == 2) {
        if (use_p) fine = topp_fine<T>(row, rowflat, V, P.mis, kkey, mx, cs, pp, zpre, S, pkey);
    }
    if (use_p && !fine) {
        // Top-p within the top-k set: the fewest value levels from the top holding top_p of its
        // mass; the top digit's mass histogram over the set also gives the set's total.
        double target = 0.0;
        uint32_t prefix = 0u;
        for (int lvl = 0; lvl < LV; ++lvl) {
            key_histogram<T, true>(row, rowflat, V, P.mis, prefix, lvl, kkey, mx, cs, S);
            if (lvl == 0) {
                if (warp == 0) {
                    double z = 0.0;
                    for (int i = lane; i < TK_BINS; i += 32) z += S.mass[i];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
                    if (lane == 0) S.above_mass = z;
                }
                __syncthreads();
                target = (double)pp * S.above_mass;
                __syncthreads();
            }
            if (warp == 0) walk_bins(S, TK_BINS, true, 0, target, lane);
            __syncthreads();
            prefix |= (uint32_t)S.sel << KeyOf<T>::shift(lvl);
            target -= S.above_mass;
            __syncthreads();
        }
        pkey = prefix > kkey ? prefix : kkey;
    }
    if (tid == 0) P.thr[r] = KeyOf<T>::value(pkey);
    __syncthreads();
}

// A few CTAs per SM, each taking rows in turn, so that the rows being filtered at any time fit in
// L2 and a row's later passes are served from it.
// after_ring: the ring kernel ran first; only the rows it left TK_PENDING are taken.
template <typename T>
__global__ void __launch_bounds__(NT_TK, TK_CTAS) sv_topkp_kernel(const Params P, int after_ring)
{
    __shared__ TopkpSmem S;
    const int64_t R = (int64_t)P.B * P.rpr;
    pdl_launch_dependents();
    if (after_ring) pdl_wait();  // the ring grid's thresholds (a no-op unless launched as a dependent)
    for (int64_t r = blockIdx.x; r < R; r += gridDim.x) {
        if (after_ring && __float_as_uint(__ldcg(P.thr + r)) != TK_PENDING) continue;
        topkp_row<T>(P, r, S);
    }
}

}  // namespace sv
