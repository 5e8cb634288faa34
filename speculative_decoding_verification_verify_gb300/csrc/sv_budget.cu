// sv_budget.cu -- the adaptive verification budget: which draft slots of a batch to verify
// ("The speculative decoding zoo", section "The finer loop: DSpark's confidence budget": every
// (request, position) slot scores the running product of its request's confidences, a global
// top-k admits the best slots with earlier positions first on ties, and the budget maximises
// expected accepted tokens per unit of step cost; "Inference Systems Frontier: new models and
// speculative decoding", section "Deciding how much to verify by load").
//
// One kernel: a cluster of CL = 8 CTAs of 1024 threads that share their shared memory
// (distributed shared memory), n = B * K <= 16384 slots, CTA c owning slots [c 2048, c 2048 + 2048):
//   1. Survival products (fp32, the precision the decision is taken in) and sort keys ~bits(score),
//      whose ascending order is descending score; slots past a request's draft count, and past n,
//      take the key of a zero score.  Each CTA sorts its 2048 keys: blocks of 64 by a bitonic
//      network in registers, then five merge-path rounds in shared memory.
//   2. The batch's sorted order, by three rounds of merging: round L merges, in every group of 2^L
//      CTAs, the sorted sequences of its two halves, each CTA writing its own 2048 positions of the
//      group's merge.  The merge path gives the two ends of that slice (a 32-way search by one warp
//      in the other CTAs' keys), the two pieces between them are copied in, and each thread merges
//      two positions (one merge-path search in the local copies).  Equal keys: the lower half's
//      first.  CTA c ends with positions [c 2048, c 2048 + 2048) of the sorted order.  Equal
//      scores come out in some order: the gains depend only on the values, and admission orders
//      ties as the rule does.
//   3. gain[b] = the sum of the b best scores, a scan in 64-bit fixed point (units of 2^-49: exact
//      for scores >= 2^-26, the rest truncated by less than 2^-49 each, so B + gain is within
//      64 * 2^-49 ~ 1e-13 of exact relative to B, as n <= 64 B); the rate (B + gain[b]) / cost[b]
//      of every budget as a 64-bit key (exponent, then 47 mantissa bits; relative error below
//      2^-45) computed in fp32 double-float arithmetic, and the first maximum of the keys: in each
//      CTA, then over the eight CTAs.  Rates within about 2^-44 of each other may come out in
//      either order.  No fp64 arithmetic: GB300 has few fp64 units, and a chain of fp64
//      comparisons run by every thread cost microseconds.
//   4. The admitted prefix of each request: its slots scoring above the chosen budget's last score
//      s*, then its slots scoring s* in the rule's tie order (position, then request) while the
//      budget lasts.
#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "spec_verify.h"
#include "sv_check.cuh"

namespace svb {

namespace cg = cooperative_groups;

constexpr int MAX_SLOTS = SPEC_VERIFY_BUDGET_MAX_SLOTS;
constexpr int MAX_K = 64;
constexpr int CL = 8;                 // CTAs of the cluster
constexpr int NT = 1024;
constexpr int NW = NT / 32;
constexpr int PER = MAX_SLOTS / CL;   // slots of a CTA
constexpr int KPT = PER / NT;         // slots of a thread
constexpr uint32_t ZERO_KEY = 0xffffffffu;  // ~bits(+0): the last key; also the padding
constexpr int FIX_SHIFT = 49;
constexpr int LOG_PER = 11;
static_assert(PER == 1 << LOG_PER, "a CTA's slots: a power of two");

struct PlanSmem {
    uint32_t loc[PER];          // this CTA's keys sorted locally; later the second merge round's output
    uint32_t orig[PER];         // the same keys in slot order (request-major)
    uint32_t fin[PER];          // the first and third merge rounds' output: at the end, this CTA's
                                //  slice of the batch's sorted order
    union {
        float cf[PER + 2 * MAX_K];  // the confidences of the requests touching this CTA's slots
        uint32_t tmp[PER];          // a merge round's two pieces
    };
    double cst[PER];            // cost[s0 + x + 1]: the costs of this CTA's budgets
    double cost0;               // cost[0] (CTA 0)
    int nd[PER + 2];            // num_drafts of the requests touching this CTA's slots, as given
    unsigned long long wsum[NW];
    unsigned long long wkey[NW];  // the warps' best rate keys ...
    int wbud[NW];                 // ... and budgets
    int wcnt[NW];
    int split[2];               // a merge round's split at this slice's two ends
    int lohi[2];                // valid keys below s*'s key, at or below it
    // Written by every CTA q of the cluster into slot q (stored ahead of a cluster barrier, so that
    // after it each CTA reads its own copy):
    unsigned long long tot_in[CL];  // fixed-point sums of the CTAs' slices (valid positions)
    unsigned long long key_in[CL];  // the CTAs' best rate keys ...
    int bud_in[CL];                 // ... budgets ...
    uint32_t skey_in[CL];           // ... and the keys at those budgets' last positions
    // Published to the cluster:
    int nvalid;
};

__device__ __forceinline__ float score_of_key(uint32_t k) { return __uint_as_float(~k); }

// A score in [0, 1] in units of 2^-49, rounded down: the mantissa shifted by the exponent.
__device__ __forceinline__ unsigned long long fixed49(float v)
{
    const uint32_t u = __float_as_uint(v);
    const int ex = (int)(u >> 23) - 127;
    if (!(v > 0.f) || ex < -49) return 0ull;
    const unsigned long long m = (u & 0x7fffffu) | 0x800000u;
    const int sh = ex + FIX_SHIFT - 23;
    return sh >= 0 ? m << sh : m >> (-sh);
}

constexpr int KEY_BIAS = 2048;  // rate keys: the binary exponent E + KEY_BIAS above 47 mantissa bits

// An fp32 value of the 24 bits of m below its top bit (which sits at bit `top`), scaled into
// [0, 2^-23) -- the low word of a double-float whose high word holds the top 24 bits.
__device__ __forceinline__ float low24(unsigned long long m, int top)
{
    return (float)(uint32_t)((m >> (top - 47)) & 0xffffffu) * 0x1p-47f;
}

// A sortable key of the rate N / c, N = nfix 2^-48 (0 < nfix < 2^63), c a double: the rate is
// M 2^(E - 47) with M in [2^47, 2^48), and the key ((E + KEY_BIAS) << 47) | (M - 2^47) orders as
// the rates do wherever they differ by more than about 2^-44 (relative error below 2^-45).  N and
// c's mantissa are cut to 48 bits as fp32 pairs hi + lo (double-float numbers), divided by one
// correctly rounded fp32 division, whose remainder nh - qh ch is exact under an fma, and one
// correction step.  A cost that is not positive and finite gives key 0.  No fp64 arithmetic:
// GB300 has few fp64 units.
__device__ __forceinline__ unsigned long long rate_key(unsigned long long nfix, double c)
{
    const unsigned long long cb = (unsigned long long)__double_as_longlong(c);
    int ec = (int)((cb >> 52) & 0x7ff);
    unsigned long long mc = cb & ((1ull << 52) - 1);
    if ((cb >> 63) || ec == 0x7ff || (ec == 0 && mc == 0)) return 0ull;
    if (ec == 0) {  // subnormal: bring the top bit to bit 52
        const int sh = __clzll((long long)mc) - 11;
        mc = (mc << sh) & ((1ull << 52) - 1);
        ec = 1 - sh;
    }
    mc |= 1ull << 52;
    const float ch = __uint_as_float(0x3f800000u | (uint32_t)((mc >> 29) & 0x7fffffu)), cl = low24(mc, 52);
    const int lz = __clzll((long long)nfix);
    const unsigned long long m = nfix << lz;  // top bit at 63: N = (m 2^-63) 2^(15 - lz)
    const float nh = __uint_as_float(0x3f800000u | (uint32_t)((m >> 40) & 0x7fffffu)), nl = low24(m, 63);
    const float qh = __fdiv_rn(nh, ch);
    const float r = fmaf(-qh, ch, nh) + fmaf(-qh, cl, nl);
    const float ql = __fdividef(r, ch);
    long long M = (long long)(qh * 0x1p47f) + __float2ll_rn(ql * 0x1p47f);  // the quotient 2^47, in (2^46, 2^48)
    int E = (15 - lz) - (ec - 1023);
    const int s = __clzll(M) - 16;  // normalise M into [2^47, 2^48)
    M = s >= 0 ? M << s : M >> -s;
    E -= s;
    E = min(max(E + KEY_BIAS, 1), 4095);
    return ((unsigned long long)E << 47) | ((unsigned long long)M & ((1ull << 47) - 1));
}

// The double nearest the rate a key stands for (to 48 bits), by its bits.
__device__ __forceinline__ double rate_of_key(unsigned long long key)
{
    if (key == 0ull) return 0.0;
    const int be = (int)(key >> 47) - KEY_BIAS + 1023;  // the double's biased exponent
    if (be <= 0) return 0.0;
    if (be >= 2047) return __longlong_as_double(0x7ff0000000000000ll);
    return __longlong_as_double((long long)(((unsigned long long)be << 52) | ((key & ((1ull << 47) - 1)) << 5)));
}

// The first maximum: does budget a with key ka come before budget b with key kb?
__device__ __forceinline__ bool beats(unsigned long long ka, int a, unsigned long long kb, int b)
{
    return ka > kb || (ka == kb && a < b);
}

__device__ __forceinline__ float clip01(float c) { return fminf(fmaxf(c, 0.f), 1.f); }  // NaN reads as 0
__device__ __forceinline__ uint32_t key_of(float run) { return ~(__float_as_uint(run) & 0x7fffffffu); }

// Block-wide sum of one int per thread (every thread of the CTA calls it).
__device__ __forceinline__ int block_sum(int x, int lane, int warp, int *ws)
{
    x = __reduce_add_sync(0xffffffffu, x);
    __syncthreads();
    if (lane == 0) ws[warp] = x;
    __syncthreads();
    int t = 0;
    for (int w = 0; w < NW; ++w) t += ws[w];
    return t;
}

// Block-wide exclusive scan of one int per thread; *total = the sum.
__device__ __forceinline__ int block_excl_scan(int x, int lane, int warp, int *ws, int &total)
{
    int incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    __syncthreads();
    if (lane == 31) ws[warp] = incl;
    __syncthreads();
    int before = incl - x;
    total = 0;
    for (int w = 0; w < NW; ++w) {
        if (w < warp) before += ws[w];
        total += ws[w];
    }
    return before;
}

// Global-to-shared copies that do not pass through registers, so that all of a thread's loads are
// in flight at once; cp_async_wait() waits for this thread's.
__device__ __forceinline__ void cp_async4(void *dst, const void *src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async8(void *dst, const void *src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// The first index in [lo, hi] at which the predicate f (true on a prefix, then false) is false,
// f(hi) taken as false: one warp, each round probing 32 evenly spaced points (f is evaluated only
// below hi) and keeping the interval between the last true and the first false probe.  A range of
// 16385 takes three rounds.
template <class F>
__device__ __forceinline__ int warp_first_false(int lo, int hi, int lane, F f)
{
    while (hi > lo) {
        const int step = (hi - lo + 31) >> 5;
        const int p = lo + (lane + 1) * step - 1;
        const int t = __popc(__ballot_sync(0xffffffffu, p < hi && f(p)));
        lo += t * step;
        hi = min(hi, lo + step - 1);
    }
    return lo;
}

// One compare-exchange of a bitonic stage: elements e (this lane's x) and e ^ j (the partner's y),
// ascending where (e & k) == 0.
__device__ __forceinline__ uint32_t cx(uint32_t x, uint32_t y, int e, int j, int k)
{
    const bool low = (e & j) == 0, asc = (e & k) == 0;
    return (low == asc) ? min(x, y) : max(x, y);
}

// Merge-path output of positions d and d + 1 of the merge of sorted ta[0, la) and tb[0, lb)
// (d + 1 < la + lb; ta's keys first on ties) into out[d], out[d + 1]: the count of ta's keys among
// the first d is the first a at which ta[a] <= tb[d - a - 1] fails.
__device__ __forceinline__ void merge_two(const uint32_t *ta, int la, const uint32_t *tb, int lb, int d,
                                          uint32_t *out)
{
    int lo = max(0, d - lb), hi = min(d, la);
    while (lo < hi) {
        const int m = (lo + hi) >> 1;
        if (ta[m] <= tb[d - m - 1]) lo = m + 1;
        else hi = m;
    }
    int ia = lo, ib = d - lo;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const bool take_a = ia < la && (ib >= lb || ta[ia] <= tb[ib]);
        out[d + e] = take_a ? ta[ia++] : tb[ib++];
    }
}

// Ascending sort of loc[0, PER) by NT threads, through tmp: blocks of 64 by a bitonic network in
// registers (thread t holds elements 2t and 2t + 1, the stages across a warp by shuffles; the last
// phase sorts every block ascending), then five merge-path rounds double the sorted blocks up to
// PER, two positions per thread.
__device__ __forceinline__ void local_sort(uint32_t *loc, uint32_t *tmp, int tid)
{
    static_assert(PER == 2 * NT, "two elements per thread");
    uint32_t v0 = loc[2 * tid], v1 = loc[2 * tid + 1];
#pragma unroll
    for (int k = 2; k <= 64; k <<= 1) {
        const int kd = k == 64 ? PER : k;  // the direction bit of element e is e & kd
#pragma unroll
        for (int j = k >> 1; j >= 2; j >>= 1) {
            const int m = j >> 1;  // partner lane: lane ^ m (elements 2t + h and (2t + h) ^ j)
            const uint32_t y0 = __shfl_xor_sync(0xffffffffu, v0, m), y1 = __shfl_xor_sync(0xffffffffu, v1, m);
            v0 = cx(v0, y0, 2 * tid, j, kd);
            v1 = cx(v1, y1, 2 * tid + 1, j, kd);
        }
        const bool asc = ((2 * tid) & kd) == 0;  // j == 1: within the thread
        const uint32_t lo = min(v0, v1), hi = max(v0, v1);
        v0 = asc ? lo : hi;
        v1 = asc ? hi : lo;
    }
    tmp[2 * tid] = v0;
    tmp[2 * tid + 1] = v1;
    uint32_t *src = tmp, *dst = loc;
    for (int w = 64; w < PER; w <<= 1) {  // five rounds: tmp -> loc -> tmp -> loc -> tmp -> loc
        __syncthreads();
        const int base = (2 * tid) & ~(2 * w - 1);
        merge_two(src + base, w, src + base + w, w, 2 * tid - base, dst + base);
        uint32_t *t = src;
        src = dst;
        dst = t;
    }
    __syncthreads();
}

__global__ void __cluster_dims__(CL, 1, 1) __launch_bounds__(NT, 1)
    plan_kernel(const float *conf, const int32_t *num_drafts, int B, int K, const double *cost, int32_t *admitted,
                int32_t *budget_out, double *rate_out)
{
    extern __shared__ __align__(16) unsigned char plan_raw[];
    PlanSmem &S = *reinterpret_cast<PlanSmem *>(plan_raw);
    cg::cluster_group cluster = cg::this_cluster();
    const int c = (int)cluster.block_rank();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n = B * K;
    auto drafts_of = [&](int r) { return num_drafts ? min(max(num_drafts[r], 0), K) : K; };
    auto peer = [&](auto *p, int rank) { return cluster.map_shared_rank(p, rank); };
    // 1. Keys of slots [s0, s1).  Staged first, all in flight together: the confidences of the
    // requests touching them, their draft counts, and the costs of this CTA's budgets.
    const int s0 = c * PER, s1 = min(s0 + PER, n);
    const int r0 = s0 < n ? s0 / K : 0, r1 = s1 > s0 ? (s1 - 1) / K + 1 : 0;  // requests [r0, r1)
    const int c0 = r0 * K, nc = r1 > r0 ? min(r1 * K, n) - c0 : 0;
    for (int j = tid; j < nc; j += NT) {
        if (SV_INB(c0 + j, n, 901)) cp_async4(&S.cf[j], conf + c0 + j);
        else S.cf[j] = 0.f;
    }
    if (num_drafts)
        for (int r = r0 + tid; r < r1; r += NT) cp_async4(&S.nd[r - r0], num_drafts + r);
    for (int x = tid; x < PER; x += NT) {
        if (s0 + x + 1 <= n) cp_async8(&S.cst[x], cost + s0 + x + 1);
        else S.cst[x] = 1.0;
        S.loc[x] = ZERO_KEY;
    }
    if (c == 0 && tid == 0) cp_async8(&S.cost0, cost);
    cp_async_wait();
    __syncthreads();
    auto nd_of = [&](int r) { return num_drafts ? min(max(S.nd[r - r0], 0), K) : K; };  // r in [r0, r1)
    int my_valid = 0;
    for (int r = r0 + tid; r < r1; r += NT) {
        const int nd = nd_of(r);
        float run = 1.f;
        for (int i = 0; i < nd; ++i) {
            run = run * clip01(S.cf[(r - r0) * K + i]);
            const int j = r * K + i;
            if (j >= s0 && j < s1) {
                S.loc[j - s0] = key_of(run);
                ++my_valid;
            }
        }
    }
    const int part_valid = block_sum(my_valid, lane, warp, S.wcnt);
    for (int x = tid; x < PER; x += NT) S.orig[x] = S.loc[x];
    if (tid == 0) S.nvalid = part_valid;
    local_sort(S.loc, S.tmp, tid);  // the confidences' staging area is free again
    cluster.sync();  // #1: every CTA's sorted keys and valid count are visible
    int nvq[CL];
#pragma unroll
    for (int q = 0; q < CL; ++q) nvq[q] = *peer(&S.nvalid, q);  // loads in flight together
    int nv = 0;
#pragma unroll
    for (int q = 0; q < CL; ++q) nv += nvq[q];
    // 2. Merge rounds L = 1, 2, 3: in each group of 2^L CTAs (from g0), the halves' sorted
    // sequences A (CTAs g0 ..) and B (the rest), half PER keys each, merged into dst; this CTA
    // writes positions [d0, d0 + PER) of the group's merge, d0 = (c - g0) PER.  The merge path at
    // diagonal d: the count a of A's keys among the merge's first d, the first a at which
    // A[a] <= B[d - a - 1] fails (A's keys first on ties).  The last round also sums this CTA's
    // slice (3., below), so that the round's cluster barrier publishes the total.
    const int xb = tid * KPT;  // this thread's positions [xb, xb + KPT): those it merges in
    unsigned long long before = 0ull;  // fixed-point sum of the valid positions before xb
    for (int L = 1; L <= 3; ++L) {
        const uint32_t *src = L == 2 ? S.fin : S.loc;
        uint32_t *dst = L == 2 ? S.loc : S.fin;
        const int half = 1 << (L - 1), g0 = c & ~(2 * half - 1), na = half * PER;
        auto key_a = [&](int i) { return *peer(&src[i & (PER - 1)], g0 + (i >> LOG_PER)); };
        auto key_b = [&](int i) { return *peer(&src[i & (PER - 1)], g0 + half + (i >> LOG_PER)); };
        const int d0 = (c - g0) * PER;
        if (warp < 2) {  // warp 0: the split at d0; warp 1: at d0 + PER
            const int d = d0 + warp * PER;
            const int a = warp_first_false(max(0, d - na), min(d, na), lane,
                                           [&](int p) { return key_a(p) <= key_b(d - p - 1); });
            if (lane == 0) S.split[warp] = a;
        }
        __syncthreads();
        const int a0 = S.split[0], la = S.split[1] - a0, b0 = d0 - a0;
        for (int e = tid; e < PER; e += NT) {
            const bool in_a = e < la;
            const int i = in_a ? a0 + e : b0 + (e - la);
            S.tmp[e] = SV_INB(i, na, 907) ? (in_a ? key_a(i) : key_b(i)) : ZERO_KEY;
        }
        __syncthreads();
        merge_two(S.tmp, la, S.tmp + la, PER - la, xb, dst);
        if (L == 3) {
            // 3. The fixed-point sum of this CTA's slice, and of the valid positions before xb.
            unsigned long long own = 0ull;
#pragma unroll
            for (int u = 0; u < KPT; ++u)
                if (s0 + xb + u < nv) own += fixed49(score_of_key(dst[xb + u]));
            unsigned long long incl = own;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            if (lane == 31) S.wsum[warp] = incl;
            __syncthreads();
            static_assert(NW == 32, "one warp sum per lane");
            const unsigned long long ws = S.wsum[lane];
            unsigned long long wincl = ws;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned long long y = __shfl_up_sync(0xffffffffu, wincl, o);
                if (lane >= o) wincl += y;
            }
            before = incl - own + __shfl_sync(0xffffffffu, wincl - ws, warp);
            const unsigned long long ctot = __shfl_sync(0xffffffffu, wincl, 31);
            if (tid < CL) *peer(&S.tot_in[c], tid) = ctot;
        }
        cluster.sync();  // the round's slices (and the totals) are complete, its sources no longer read
    }
    for (int q = 0; q < c; ++q) before += S.tot_in[q];
    // Gains of this CTA's positions g = s0 + x (budget b = g + 1), their rates' keys, and the first
    // maximum: of this thread's budgets, of the CTA's (shuffles, then one warp over the warps'),
    // and of the cluster's (every CTA reduces the eight CTAs' bests the same way, so all agree).
    // The cost of budget b, for b = 0 (CTA 0) and this CTA's budgets [s0 + 1, s0 + PER].
    auto cost_of = [&](int b) { return b == 0 ? S.cost0 : SV_INB(b - s0 - 1, PER, 903) ? S.cst[b - s0 - 1] : 1.0; };
    const unsigned long long bfix = (unsigned long long)B << (FIX_SHIFT - 1);  // B in units of 2^-48
    unsigned long long bkey = 0ull;
    int bbud = 0x7fffffff;
    {
        unsigned long long g = before;
#pragma unroll
        for (int u = 0; u < KPT; ++u) {
            const int b = s0 + xb + u + 1;
            if (b > nv) break;
            g += fixed49(score_of_key(S.fin[xb + u]));
            const unsigned long long k = rate_key(bfix + (g >> 1), cost_of(b));
            if (beats(k, b, bkey, bbud)) {
                bkey = k;
                bbud = b;
            }
        }
        if (c == 0 && tid == 0) {  // budget 0
            const unsigned long long k = rate_key(bfix, cost_of(0));
            if (beats(k, 0, bkey, bbud)) {
                bkey = k;
                bbud = 0;
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long ok = __shfl_xor_sync(0xffffffffu, bkey, o);
        const int ob = __shfl_xor_sync(0xffffffffu, bbud, o);
        if (beats(ok, ob, bkey, bbud)) {
            bkey = ok;
            bbud = ob;
        }
    }
    if (lane == 0) {
        S.wkey[warp] = bkey;
        S.wbud[warp] = bbud;
    }
    __syncthreads();
    if (warp == 0) {
        bkey = S.wkey[lane];
        bbud = S.wbud[lane];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const unsigned long long ok = __shfl_xor_sync(0xffffffffu, bkey, o);
            const int ob = __shfl_xor_sync(0xffffffffu, bbud, o);
            if (beats(ok, ob, bkey, bbud)) {
                bkey = ok;
                bbud = ob;
            }
        }
        // The best budget's last position, b - 1, is this CTA's when b is in [s0 + 1, s0 + PER]
        // (b is 0, or past the range when this CTA has no valid budget).
        const uint32_t sk = bbud > s0 && bbud <= s0 + PER ? S.fin[bbud - 1 - s0] : 0u;
        if (lane < CL) {
            *peer(&S.key_in[c], lane) = bkey;
            *peer(&S.bud_in[c], lane) = bbud;
            *peer(&S.skey_in[c], lane) = sk;
        }
    }
    cluster.sync();  // #2: the CTAs' bests
    int budget = S.bud_in[0], win = 0;
    bkey = S.key_in[0];
    for (int q = 1; q < CL; ++q)
        if (beats(S.key_in[q], S.bud_in[q], bkey, budget)) {
            bkey = S.key_in[q];
            budget = S.bud_in[q];
            win = q;
        }
    if (c == 0 && tid == 0) {
        *budget_out = budget;
        if (rate_out) *rate_out = rate_of_key(bkey);
    }
    // s*: the key at sorted position budget - 1 (sent by its owner with its best); the valid slots
    // scoring above it and at it, counted in the batch's sorted keys G: warp 0 the keys below s*'s
    // key (budget - 1 unless G[budget - 2] ties it), warp 1 those at or below it (budget unless
    // G[budget] ties it); a tie is resolved by a search over the positions past the neighbour.
    const uint32_t skey = budget > 0 ? S.skey_in[win] : 0u;
    if (warp < 2) {
        int cnt = 0;
        if (budget > 0) {
            auto key_g = [&](int i) { return *peer(&S.fin[i & (PER - 1)], i >> LOG_PER); };
            if (warp == 0) {
                cnt = budget - 1;
                if (cnt > 0 && !(key_g(cnt - 1) < skey))
                    cnt = warp_first_false(0, cnt - 1, lane, [&](int i) { return key_g(i) < skey; });
            } else {
                cnt = budget;
                if (cnt < CL * PER && key_g(cnt) <= skey)
                    cnt = warp_first_false(cnt + 1, CL * PER, lane, [&](int i) { return key_g(i) <= skey; });
            }
        }
        if (lane == 0) S.lohi[warp] = cnt;
    }
    __syncthreads();
    const int above = S.lohi[0];
    // The padding shares the zero key: ties of a zero s* are the valid zero scores.
    const int ties = budget <= 0 ? 0 : skey == ZERO_KEY ? nv - above : S.lohi[1] - above;
    // 4. Admission.  Request r is handled by the CTA owning its first slot; its keys are read from
    // the slot-order copies (the next CTA's for slots past this CTA's range).
    auto key_at = [&](int j) { return j < s1 ? S.orig[j - s0] : *peer(&S.orig[(j - s0) - PER], c + 1); };
    const int ra = (s0 + K - 1) / K, rb = s1 > s0 ? (s1 - 1) / K + 1 : ra;  // requests starting here
    const int need = budget - above;  // tie slots admitted (1 <= need <= ties when budget > 0)
    if (budget <= 0 || need >= ties) {
        for (int r = ra + tid; r < rb; r += NT) {
            int a = 0;
            if (budget > 0) {
                const int nd = nd_of(r);
                for (int i = 0; i < nd; ++i) a += key_at(r * K + i) <= skey;
            }
            admitted[r] = a;
        }
    } else if (c == 0) {
        // Part of the tie group: position by position, requests in order (a block scan per chunk
        // of NT requests), the tie slots ranked below `need` admitted.  CTA 0 alone.
        auto key_any = [&](int j) { return *peer(&S.orig[j % PER], j / PER); };
        auto gt_eq = [&](int r, int &gt, int &eq) {
            gt = 0;
            eq = 0;
            const int nd = drafts_of(r);
            for (int i = 0; i < nd; ++i) {
                const uint32_t x = key_any(r * K + i);
                gt += x < skey;
                eq += x == skey;
            }
        };
        const int chunks = (B + NT - 1) / NT;
        for (int m = 0; m < chunks; ++m) {
            const int r = m * NT + tid;
            if (r < B) {
                int gt, eq;
                gt_eq(r, gt, eq);
                admitted[r] = gt;
            }
        }
        int tie_base = 0;
        for (int i = 0; i < K; ++i) {
            for (int m = 0; m < chunks; ++m) {
                const int r = m * NT + tid;
                int gt = 0, eq = 0;
                if (r < B) gt_eq(r, gt, eq);
                const int is_tie = r < B && i >= gt && i < gt + eq;
                int total;
                const int rank = tie_base + block_excl_scan(is_tie, lane, warp, S.wcnt, total);
                if (is_tie && rank < need) admitted[r] = i + 1;
                tie_base += total;
            }
        }
    }
    cluster.sync();  // #3: no CTA leaves while another may still read its shared memory
}

}  // namespace svb

namespace sv {
// This module's first range violation (debug builds; 0 otherwise), cleared when read.
unsigned long long budget_debug_fault()
{
#ifdef SV_DEBUG
    unsigned long long w = 0, z = 0;
    if (cudaMemcpyFromSymbol(&w, g_sv_debug_fault, sizeof w) != cudaSuccess ||
        cudaMemcpyToSymbol(g_sv_debug_fault, &z, sizeof z) != cudaSuccess)
        return ~0ull;
    return w;
#else
    return 0;
#endif
}
}  // namespace sv

extern "C" size_t spec_verify_plan_budget_workspace_bytes(int B, int K)
{
    if (B < 1 || K < 1 || K > svb::MAX_K || (int64_t)B * K > svb::MAX_SLOTS) return 0;
    return 256;  // reserved: the planner keeps its work in shared memory
}

static std::mutex g_plan_mu;
static bool g_plan_attr[64];

extern "C" int spec_verify_plan_budget(const float *conf, const int32_t *num_drafts, int B, int K,
                                       const double *cost, int32_t *admitted, int32_t *budget,
                                       double *best_rate, void *workspace, size_t ws_bytes, void *stream)
{
    if (!conf || !cost || !admitted || !budget || !workspace) return SPEC_VERIFY_EINVAL;
    if (B < 1 || K < 1 || K > svb::MAX_K || (int64_t)B * K > svb::MAX_SLOTS) return SPEC_VERIFY_EINVAL;
    if ((uintptr_t)conf % 4 || (uintptr_t)cost % 8 || (uintptr_t)admitted % 4 || (uintptr_t)budget % 4 ||
        (uintptr_t)num_drafts % 4 || (uintptr_t)best_rate % 8)
        return SPEC_VERIFY_EINVAL;
    if ((uintptr_t)workspace % 8 || ws_bytes < spec_verify_plan_budget_workspace_bytes(B, K))
        return SPEC_VERIFY_EWORKSPACE;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SPEC_VERIFY_ECUDA;
    {
        std::lock_guard<std::mutex> lk(g_plan_mu);
        if (!g_plan_attr[dev]) {
            if (cudaFuncSetAttribute(svb::plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)sizeof(svb::PlanSmem)) != cudaSuccess) {
                cudaGetLastError();
                return SPEC_VERIFY_ECUDA;
            }
            g_plan_attr[dev] = true;
        }
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    svb::plan_kernel<<<svb::CL, svb::NT, sizeof(svb::PlanSmem), s>>>(conf, num_drafts, B, K, cost, admitted,
                                                                     budget, best_rate);
    return cudaGetLastError() == cudaSuccess ? SPEC_VERIFY_OK : SPEC_VERIFY_ECUDA;
}
