// sv_topkp_ring.cuh -- top-k / top-p thresholds of bf16 rows with top-k, in one read of each row.
//
// The filter is the one of sv_topkp.cuh ("投机解码", section 接受规则为什么不改变分布: p already
// carries temperature, top-k and top-p): keep every logit at or above the k-th largest, then the
// fewest whole value levels from the top whose mass, renormalised over that set, reaches top_p.
//
// Two CTAs per SM take rows in turn (while one finishes a row the other streams).  A CTA's last
// warp streams its rows, back to back, through a ring of shared-memory stages with bulk
// asynchronous copies (cp.async.bulk; a "full" mbarrier per slot counts the copy's bytes, an
// "empty" one the folding warps that have read it), so the ring's stages are in flight while the
// folding warps work, and the next row's first stages arrive while they finish the last one.
// Folding a stage, thread t takes the largest key of its group -- the stage's vectors t,
// t + NT_RING, t + 2 NT_RING, t + 3 NT_RING -- and keeps it in shared memory (2 bytes a group,
// 4008 groups for a row of 128256).  The folding warps synchronise among themselves only (named
// barrier 1), never with the copy warp.
//
// The k-th largest of the threads' maxima, L, is at most the row's k-th largest logit (the k
// largest thread maxima are k distinct logits of the row), so every logit of the top-k set lies
// in [L, max], and only groups whose largest key reaches L can hold one -- about k of the row's
// groups.  Warp 0 finds L by a binary search over the TK_SPAN keys below the maximum's (a wider
// range leaves the row to the general kernel), counting the thread maxima that reach a key with
// one warp reduction per step.  Those groups alone are read again (64 bytes each, mostly from L2)
// and every logit >= L is counted in one bin per key below the row maximum's key.  A value
// level's mass is its count times its term 2^((l - max) * cs) in 64-bit fixed point (fixed44:
// exact integer sums, no fp64 arithmetic, of which GB300 has little), and warp 0 scans the bins
// from the top for the k-th largest key and the fewest whole levels holding top_p of the top-k
// set's mass, while the other warps go on to the next row.
//
// Rows this kernel does not take -- top-k off or above NT_RING, rows longer than 32768 vectors, a
// key range [L, max] wider than TK_SPAN, or more than RING_MAX_CAND groups reaching L -- get
// TK_PENDING, and the general kernel (sv_topkp.cuh), run next, finds their thresholds.  Every
// wait on an mbarrier gives up after 0.2 s (a copy should land in microseconds): the CTA then
// leaves its current and later rows to the general kernel, so the results stay exact, waits
// (again at most 0.2 s a slot) for the last copy issued into each ring slot, and counts the event
// in the module's timeout word (spec_verify_wait_timeouts).
#pragma once

#include "sv_topkp.cuh"

namespace sv {

#ifndef SV_RING_STAGE_VEC
#define SV_RING_STAGE_VEC 1024
#endif
#ifndef SV_RING_STAGES
#define SV_RING_STAGES 5
#endif
#ifndef SV_RING_CTAS
#define SV_RING_CTAS 2
#endif
#ifndef SV_RING_NT
#define SV_RING_NT 256
#endif
constexpr int NT_RING = SV_RING_NT;                      // folding threads per CTA (plus one copy warp)
constexpr int RING_STAGE_VEC = SV_RING_STAGE_VEC;        // 16-byte vectors per stage (16 KB)
constexpr int RING_STAGES = SV_RING_STAGES;              // stages of the ring (80 KB)
constexpr int RING_CTAS = SV_RING_CTAS;                  // CTAs per SM
constexpr int RING_GV = RING_STAGE_VEC / NT_RING;        // vectors of one thread's group in a stage
constexpr int RING_MAX_ST = 32768 / RING_STAGE_VEC;      // stages of a row at most (rows up to 262158)
constexpr int RING_MAX_CAND = 1024;                      // groups pass 2 reads again, at most
constexpr unsigned long long RING_WAIT_NS = 200000000ull;

// Stage waits that ran out of time since the module was loaded.
static __device__ unsigned long long g_ring_timeouts;

struct RingSmem {
    uint4 ring[RING_STAGES][RING_STAGE_VEC];
    int cnt[TK_SPAN];                       // one bin per key below the row maximum's key
    uint16_t gkey[RING_MAX_ST][NT_RING];    // largest key of group (stage, thread)
    uint32_t tkey[NT_RING];                 // each thread's largest key
    uint32_t cand[RING_MAX_CAND];           // pass 2's groups: stage << 16 | thread
    unsigned long long full[RING_STAGES];   // a stage has landed (the copy's bytes)
    unsigned long long empty[RING_STAGES];  // every folding warp has read the stage
    float wmax[NT_RING / 32];
    uint32_t wkey[NT_RING / 32];
    int abort, issued;                      // a wait ran out; stages the copy warp issued
    int status;                             // warp 0's verdict on the row (see ring_fold_rows)
    int ncand;                              // pass 2's groups listed
    uint32_t lkey, mkey;                    // L's key and the row maximum's
};

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(unsigned long long *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Makes the barriers' initialisation visible to the copy engine.
__device__ __forceinline__ void mbar_init_fence()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Orders this CTA's earlier shared-memory accesses before later asynchronous copies into it.
__device__ __forceinline__ void async_proxy_fence()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

#ifndef SV_RING_EF
#define SV_RING_EF 1
#endif
// bytes (a multiple of 16, both addresses 16-byte aligned) from global src to shared dst; the
// stage's barrier completes its phase when they have landed.  The lines are read once (the
// streaming pass that follows reads every row again, but 128 MB rows do not survive in L2 from
// one pass to the next), so with SV_RING_EF they enter L2 at evict-first priority and leave the
// rest of its contents alone.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, unsigned long long *bar)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
#if SV_RING_EF
    unsigned long long pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
#else
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
#endif
}

__device__ __forceinline__ bool mbar_try_wait(unsigned long long *bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ unsigned long long global_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

#ifndef SV_RING_SPIN_NS
#define SV_RING_SPIN_NS 0
#endif
// Wait for the phase of the given parity to complete; false after RING_WAIT_NS.  Between polls a
// waiting warp sleeps SV_RING_SPIN_NS, leaving the issue slots to the warps that work.
__device__ __forceinline__ bool mbar_wait(unsigned long long *bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (SV_RING_SPIN_NS > 0) __nanosleep(SV_RING_SPIN_NS);
        if (global_ns() - t0 > RING_WAIT_NS) return false;
    }
    return true;
}

// A term in units of 2^-44 of the row maximum's term (see fixed_term): a row's masses, count times
// term summed over levels, stay below 2^63 for rows of up to 2^19 logits, and the sums are exact;
// the top-p crossing is placed within about 1e-8 of the row maximum's term.
__device__ __forceinline__ unsigned long long fixed44(float t) { return fixed_term(t, 44); }

// What becomes of row r: kind 0 not filtered (threshold -inf), 1 this kernel, 2 the general one.
struct RingRow {
    int kind, kk, nst, nx;  // kind, top-k, stages, elements outside the aligned body (< 16)
    float pp, cs;
    bool use_p;
    int64_t a0, nv;  // the body: first element (16-byte aligned) and its 16-byte vectors
};

__device__ __forceinline__ RingRow ring_row(const Params &P, int64_t r)
{
    RingRow w{};
    const int b = (int)(r / P.rpr);
    const int64_t V = P.V;
    w.kind = 2;
    if (!(SV_INB(b, P.B, 721) && SV_INB(r, (int64_t)P.B * P.rpr, 722))) return w;
    const float Tb = P.temps ? __ldg(P.temps + b) : 1.f;
    w.kk = P.top_k ? __ldg(P.top_k + b) : 0;
    w.pp = P.top_p ? __ldg(P.top_p + b) : 1.f;
    const bool use_k = w.kk >= 1 && (int64_t)w.kk < V;
    w.use_p = w.pp < 1.f;
    if (Tb == 0.f || (!use_k && !w.use_p)) {
        w.kind = 0;
        return w;
    }
    w.cs = P.temps ? cs_of(Tb) : P.cs;
    w.a0 = min((int64_t)((8 - (r * V + P.mis) % 8) % 8), V);
    w.nv = (V - w.a0) / 8;
    if (!use_k || w.kk > NT_RING || w.nv > (int64_t)RING_MAX_ST * RING_STAGE_VEC) return w;
    w.nst = (int)((w.nv + RING_STAGE_VEC - 1) / RING_STAGE_VEC);
    w.nx = (int)(V - w.nv * 8);
    w.kind = 1;
    return w;
}

// The copy warp's cursor: the row it is copying, its next stage, and the row's shape (nst < 0:
// not yet looked at).
struct RingCursor {
    int64_t r;
    int c, nst;
    int64_t a0, nv;
};

// The next stage of this CTA's rows: true with its first element and vector count, false when
// none remain.
__device__ __forceinline__ bool ring_next(const Params &P, RingCursor &cur, int64_t &e0, int &n)
{
    const int64_t R = (int64_t)P.B * P.rpr;
    while (cur.r < R) {
        if (cur.nst < 0) {
            const RingRow w = ring_row(P, cur.r);
            cur.nst = w.kind == 1 ? w.nst : 0;
            cur.a0 = w.a0;
            cur.nv = w.nv;
        }
        if (cur.c < cur.nst) {
            const int64_t v0 = (int64_t)cur.c * RING_STAGE_VEC;
            n = (int)min((int64_t)RING_STAGE_VEC, cur.nv - v0);
            e0 = cur.r * P.V + cur.a0 + v0 * 8;
            ++cur.c;
            return true;
        }
        cur.r += gridDim.x;
        cur.c = 0;
        cur.nst = -1;
    }
    return false;
}

__device__ __forceinline__ void mbar_arrive(unsigned long long *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Barriers among the NT_RING folding threads only (named barrier 1; the copy warp is not in it).
__device__ __forceinline__ void fold_sync()
{
    asm volatile("bar.sync 1, %0;" ::"n"(NT_RING) : "memory");
}

__device__ __forceinline__ int fold_sync_count(bool p)
{
    int n;
    asm volatile("{\n .reg .pred q;\n setp.ne.u32 q, %1, 0;\n bar.red.popc.u32 %0, 1, %2, q;\n}"
                 : "=r"(n)
                 : "r"((uint32_t)p), "n"(NT_RING)
                 : "memory");
    return n;
}

// Warp 0: the threshold of row r from the bins [0, span) (d = a key's distance below the
// maximum's key), lane l taking a contiguous block of them: the k-th largest key, where the
// running count reaches k, and with top-p the first whole level whose running mass (fixed point)
// reaches top_p of the top-k set's.  Lane 0 writes thr[r].
__device__ __forceinline__ void ring_scan(const Params &P, const RingSmem &S, int64_t r, const RingRow &w,
                                          uint32_t lkey, uint32_t mkey, int lane)
{
    using K = KeyOf<__nv_bfloat16>;
    const int span = (int)(mkey - lkey) + 1;
    const float mref = K::value(mkey);
    const int per = (span + 31) / 32;
    const int d0 = min(lane * per, span), d1 = min(d0 + per, span);
    auto level_mass = [&](int d, int c) -> unsigned long long {
        return c > 0 && w.use_p ? (unsigned long long)c * fixed44(ex2((K::value(mkey - (uint32_t)d) - mref) * w.cs))
                                : 0ull;
    };
    int c_own = 0;
    unsigned long long m_own = 0ull;
    for (int d = d0; d < d1; ++d) {
        const int c = S.cnt[d];
        c_own += c;
        m_own += level_mass(d, c);
    }
    int c_inc = c_own;
    unsigned long long m_inc = m_own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int yc = __shfl_up_sync(0xffffffffu, c_inc, o);
        const unsigned long long ym = __shfl_up_sync(0xffffffffu, m_inc, o);
        if (lane >= o) {
            c_inc += yc;
            m_inc += ym;
        }
    }
    const int c_before = c_inc - c_own;
    const unsigned long long m_before = m_inc - m_own;
    // The lane whose block holds the k-th crossing: dk, and the top-p target (top_p of the mass
    // through dk).
    int dk_l = INT_MAX;
    unsigned long long target = 0ull;
    if (c_before < w.kk && c_inc >= w.kk) {
        int c = c_before;
        unsigned long long m = m_before;
        for (int d = d0; d < d1; ++d) {
            const int cd = S.cnt[d];
            c += cd;
            m += level_mass(d, cd);
            if (c >= w.kk) {
                dk_l = d;
                target = (unsigned long long)((double)w.pp * (double)m);
                break;
            }
        }
    }
    const unsigned holder = __ballot_sync(0xffffffffu, dk_l != INT_MAX);
    const int dk = __reduce_min_sync(0xffffffffu, dk_l);
    int dsel = dk;
    if (w.use_p && holder) {
        target = __shfl_sync(0xffffffffu, target, __ffs(holder) - 1);
        int dp_l = INT_MAX;
        unsigned long long m = m_before;
        for (int d = d0; d < d1 && d <= dk; ++d) {
            const int c = S.cnt[d];
            m += level_mass(d, c);
            if (c > 0 && m >= target) {
                dp_l = d;
                break;
            }
        }
        dsel = min(__reduce_min_sync(0xffffffffu, dp_l), dk);
    }
    if (lane == 0) P.thr[r] = dsel == INT_MAX ? __uint_as_float(TK_PENDING) : K::value(mkey - (uint32_t)dsel);
}

// The folding warps' part: each row of the CTA in turn, its stages as the copy warp lands them.
// Three barriers a row: after pass 1 (B1), after warp 0 has found L (B2), after pass 2 (B3); warp
// 0 then scans the bins while the other warps go on to the next row.
template <typename T>
__device__ __forceinline__ void ring_fold_rows(const Params &P, RingSmem &S, int64_t R, int tid, int lane, int warp)
{
    uint32_t used = 0;
    bool live = true;  // false once a wait ran out: this CTA's remaining rows go to the general kernel
    for (int64_t r = blockIdx.x; r < R; r += gridDim.x) {
        const RingRow w = ring_row(P, r);
        if (w.kind != 1 || !live) {
            if (tid == 0) P.thr[r] = w.kind == 0 ? NEG_INF : __uint_as_float(TK_PENDING);
            continue;
        }
        const uint16_t *rowp = reinterpret_cast<const uint16_t *>(P.logits) + r * P.V;
        // The elements outside the body, one per thread; they join group (0, t).
        uint32_t xkey = 0u;
        float vmx = NEG_INF;
        if (tid < w.nx) {
            const int64_t col = tid < w.a0 ? tid : w.a0 + w.nv * 8 + (tid - w.a0);
            if (SV_INB(r * P.V + col, P.total, 725)) {
                const uint32_t bits = __ldg(rowp + col);
                xkey = KeyOf<T>::key_of_bits(bits);
                vmx = __uint_as_float(bits << 16);
            }
        }
        uint32_t tmax = xkey;  // the key of this thread's largest logit
        if (w.nst == 0) S.gkey[0][tid] = (uint16_t)xkey;
        // Pass 1: the stages as they land; each warp frees a slot as soon as it has read it.
        for (int c = 0; c < w.nst; ++c) {
            const uint32_t j = used++;
            const int s = (int)(j % RING_STAGES);
            if (!__all_sync(0xffffffffu, mbar_wait(&S.full[s], (j / RING_STAGES) & 1u))) {
                atomicExch(&S.abort, 1);
                break;
            }
            const int nvs = (int)min((int64_t)RING_STAGE_VEC, w.nv - (int64_t)c * RING_STAGE_VEC);
            uint32_t m2 = 0xff80ff80u;  // (-inf, -inf)
#pragma unroll
            for (int g = 0; g < RING_GV; ++g) {
                const int i = g * NT_RING + tid;
                if (i < nvs) {
                    const uint4 v = S.ring[s][i];
                    m2 = bmax2_nan(m2, bmax2_nan(bmax2_nan(v.x, v.y), bmax2_nan(v.z, v.w)));
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.empty[s]);
            const float gm = fmax_nan(bf_lo(m2), bf_hi(m2));
            vmx = fmax_nan(vmx, gm);
            // A zero maximum takes the key of +0, which is at least the key of any zero in the
            // group, so that no element's key exceeds its group's.
            uint32_t gk = gm == 0.f ? 0x8000u : KeyOf<T>::key_of_bits(__float_as_uint(gm) >> 16);
            if (c == 0) gk = max(gk, xkey);
            S.gkey[c][tid] = (uint16_t)gk;
            tmax = max(tmax, gk);
        }
        // The row maximum (NaN if the row holds one) and its key, per warp; the thread maxima.
        float mx = vmx;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmax_nan(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const uint32_t mkw = __reduce_max_sync(0xffffffffu, tmax);
        if (lane == 0) {
            S.wmax[warp] = mx;
            S.wkey[warp] = mkw;
        }
        S.tkey[tid] = tmax;
        fold_sync();  // B1
        if (warp == 0) {
            // Warp 0: the row maximum; L, the largest key that at least kk thread maxima reach,
            // searched within TK_SPAN keys of the maximum's; then the bins cleared.
            float m = S.wmax[0];
            uint32_t mkey = S.wkey[0];
            for (int i = 1; i < NT_RING / 32; ++i) {
                m = fmax_nan(m, S.wmax[i]);
                mkey = max(mkey, S.wkey[i]);
            }
            // 0: go on; 1: threshold -inf (the streaming pass flags the row); 2: pending; 3: a wait
            // ran out (this and the CTA's later rows pending).  Warp 0 alone reads the abort flag,
            // which the copy warp may set at any time, so that every thread takes the same branch.
            int status = 0;
            uint32_t lkey = 0u;
            if (*(volatile int *)&S.abort) {
                status = 3;
            } else if (!(m > NEG_INF) || m != m || m == POS_INF) {
                status = 1;
            } else {
                uint32_t tk[NT_RING / 32];
#pragma unroll
                for (int i = 0; i < NT_RING / 32; ++i) tk[i] = S.tkey[i * 32 + lane];
                auto reach = [&](uint32_t x) {
                    int n = 0;
#pragma unroll
                    for (int i = 0; i < NT_RING / 32; ++i) n += tk[i] >= x;
                    return (int)__reduce_add_sync(0xffffffffu, (unsigned)n);
                };
                const int dmax = (int)min((uint32_t)(TK_SPAN - 1), mkey);
                if (reach(mkey - (uint32_t)dmax) < w.kk) {
                    status = 2;
                } else {
                    int lo = 0, hi = dmax;  // at least kk thread maxima reach mkey - hi
                    while (lo < hi) {
                        const int mid = (lo + hi) >> 1;
                        if (reach(mkey - (uint32_t)mid) >= w.kk) hi = mid;
                        else lo = mid + 1;
                    }
                    lkey = mkey - (uint32_t)hi;
                    for (int i = lane; i <= hi; i += 32) S.cnt[i] = 0;
                }
            }
            if (lane == 0) {
                S.status = status;
                S.lkey = lkey;
                S.mkey = mkey;
                S.ncand = 0;
            }
        }
        fold_sync();  // B2
        const int status = S.status;
        if (status != 0) {
            if (tid == 0) P.thr[r] = status == 1 ? NEG_INF : __uint_as_float(TK_PENDING);
            if (status == 3) live = false;
            continue;
        }
        const uint32_t lkey = S.lkey, mkey = S.mkey;
        [[maybe_unused]] const int span = (int)(mkey - lkey) + 1;
        // Pass 2: the groups that reach L are listed, then read again (mostly from L2) RING_GV
        // threads a group, one vector each, so that their loads are in flight together and no
        // thread walks a long chain alone.  Every logit >= L is counted at its key; a thread's
        // head or tail element is counted by that thread.
        const int gst = w.nst > 0 ? w.nst : 1;
        for (int c = 0; c < gst; ++c)
            if (S.gkey[c][tid] >= lkey) {
                const int i = atomicAdd(&S.ncand, 1);
                if (i < RING_MAX_CAND) S.cand[i] = ((uint32_t)c << 16) | (uint32_t)tid;
            }
        fold_sync();
        const int ncand = S.ncand;
        if (ncand > RING_MAX_CAND) {  // a wide tie at L: the general kernel takes the row
            if (tid == 0) P.thr[r] = __uint_as_float(TK_PENDING);
            continue;
        }
        const uint4 *body = reinterpret_cast<const uint4 *>(rowp + w.a0);
        for (int q = tid; q < ncand * RING_GV; q += NT_RING) {
            const uint32_t e = S.cand[q / RING_GV];
            const int c = (int)(e >> 16), t = (int)(e & 0xffffu), g = q % RING_GV;
            const int64_t i = (int64_t)c * RING_STAGE_VEC + g * NT_RING + t;
            if (i >= w.nv) continue;
            if (!SV_INB(r * P.V + w.a0 + i * 8 + 7, P.total, 726)) continue;
            uint32_t k[8];
            KeyOf<T>::keys(__ldg(body + i), k);
#pragma unroll
            for (int x = 0; x < 8; ++x)
                if (k[x] >= lkey && k[x] <= mkey && SV_INB(mkey - k[x], span, 727)) atomicAdd(&S.cnt[mkey - k[x]], 1);
        }
        if (tid < w.nx && xkey >= lkey && xkey <= mkey && SV_INB(mkey - xkey, span, 728))
            atomicAdd(&S.cnt[mkey - xkey], 1);
        fold_sync();  // B3
        if (warp == 0) ring_scan(P, S, r, w, lkey, mkey, lane);
    }
}

// The rows' thresholds (bf16 logits); RING_CTAS CTAs per SM, RingSmem in dynamic shared memory.
// Warps 0 .. NT_RING/32 - 1 fold the stages and find the thresholds; the last warp copies.  Every
// row gets a threshold, -inf, or TK_PENDING.
template <typename T>
__global__ void __launch_bounds__(NT_RING + 32, RING_CTAS) sv_topkp_ring_kernel(const Params P)
{
    static_assert(sizeof(T) == 2, "the ring kernel reads bf16 logits");
    extern __shared__ __align__(16) unsigned char ring_raw[];
    RingSmem &S = *reinterpret_cast<RingSmem *>(ring_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t R = (int64_t)P.B * P.rpr;
    pdl_launch_dependents();  // the general kernel may launch; it waits for this grid to finish
    if (tid == 0) {
        for (int s = 0; s < RING_STAGES; ++s) {
            mbar_init(&S.full[s], 1);
            mbar_init(&S.empty[s], NT_RING / 32);
        }
        S.abort = 0;
        S.issued = 0;
        mbar_init_fence();
    }
    __syncthreads();
    if (warp == NT_RING / 32) {
        // The copy warp: every stage of the CTA's rows in order, each into the ring slot its
        // predecessor there has left (all folding warps arrived on the slot's empty barrier).
        if (lane == 0) {
            RingCursor cur{(int64_t)blockIdx.x, 0, -1, 0, 0};
            uint32_t q = 0;
            int64_t e0;
            int n;
            while (ring_next(P, cur, e0, n)) {
                const int s = (int)(q % RING_STAGES);
                if (q >= RING_STAGES && !mbar_wait(&S.empty[s], (q / RING_STAGES - 1) & 1u)) {
                    atomicExch(&S.abort, 1);
                    break;
                }
                if (*(volatile int *)&S.abort) break;
                if (SV_INB(e0, P.total, 723) && SV_INB(e0 + (int64_t)n * 8 - 1, P.total, 724))
                    bulk_load(S.ring[s], reinterpret_cast<const __nv_bfloat16 *>(P.logits) + e0, (uint32_t)n * 16u,
                              &S.full[s]);
                else
                    mbar_arrive(&S.full[s]);  // debug builds: an out-of-range stage is skipped
                ++q;
            }
            S.issued = q;
        }
    } else {
        ring_fold_rows<T>(P, S, R, tid, lane, warp);
    }
    __syncthreads();
    if (tid == 0 && S.abort) {
        // A wait ran out: wait (again bounded) for the last copy issued into each slot, so that no
        // copy is in flight when the CTA's shared memory is released.
        const uint32_t q = S.issued;
        for (int s = 0; s < RING_STAGES; ++s)
            if ((uint32_t)s < q) {
                const uint32_t last = (q - 1 - s) / RING_STAGES * RING_STAGES + s;
                mbar_wait(&S.full[s], (last / RING_STAGES) & 1u);
            }
        atomicAdd(&g_ring_timeouts, 1ull);
    }
}


}  // namespace sv
