// sv_rescan.cuh -- the finalising CTA draws a token from a short column range of a logit row.
//
// The finalising kernel knows which record of the streaming pass holds the crossing of the draw
// threshold t, and the mass before that record.  The record covers one streaming chunk of at most
// CHUNK_VEC 16-byte vectors (plus an unaligned head and tail), so every thread of the CTA loads
// its few vectors of that range straight into registers (one round trip, mostly L2 hits: the
// chunk was streamed a few microseconds earlier), weighs them, finds the vector where the running
// mass crosses t with a block-wide scan, and the thread holding that vector walks its elements.
#pragma once

#include <climits>

#include "sv_device.cuh"
#include "sv_draw.cuh"

namespace sv {

// Vectors of a crossing range: at most CHUNK_VEC aligned vectors plus a partial one at each end.
constexpr int RESCAN_RANGE_VEC = CHUNK_VEC + 2;

// The 16-byte vector of a row starting at column col, with the elements outside [c0, c1) read
// as -inf, element by element, so that no byte outside [c0, c1) is touched.
template <typename T>
__device__ __noinline__ uint4 load_partial(const T *row, int64_t col, int64_t c0, int64_t c1)
{
    constexpr int VEC = Elt<T>::VEC;
    uint32_t w[4];
    if (sizeof(T) == 2) {
        const unsigned short *r16 = reinterpret_cast<const unsigned short *>(row);
        for (int i = 0; i < 4; ++i) {
            const int64_t a = col + 2 * i, b = a + 1;
            const uint32_t lo = (a >= c0 && a < c1) ? __ldg(r16 + a) : 0xff80u;
            const uint32_t hi = (b >= c0 && b < c1) ? __ldg(r16 + b) : 0xff80u;
            w[i] = lo | (hi << 16);
        }
    } else {
        const uint32_t *r32 = reinterpret_cast<const uint32_t *>(row);
        for (int i = 0; i < VEC; ++i) {
            const int64_t a = col + i;
            w[i] = (a >= c0 && a < c1) ? __ldg(r32 + a) : 0xff800000u;
        }
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Weights of one vector at column col with no excluded column in it; elements outside [c0, c1),
// or below the row's top-k / top-p threshold thr, weigh 0.
template <typename T, bool FILT>
__device__ __forceinline__ void vec_weights_plain(const uint4 &w, int col, int c0, int c1, float cs,
                                                  float mc, float thr, float (&out)[Elt<T>::VEC])
{
    constexpr int VEC = Elt<T>::VEC;
    float x[VEC];
    Elt<T>::unpack(w, x);
#pragma unroll
    for (int j = 0; j < VEC; ++j) out[j] = (!FILT || x[j] >= thr) ? ex2(fmaf(x[j], cs, -mc)) : 0.f;
    if (col < c0 || col + VEC > c1) {
#pragma unroll
        for (int j = 0; j < VEC; ++j)
            if (col + j < c0 || col + j >= c1) out[j] = 0.f;
    }
}

// Rounds of the rescan: thread t weighs vectors t, t + nt, ... of the range.
constexpr int RESCAN_ROUNDS = (RESCAN_RANGE_VEC + 255) / 256;
constexpr int RESCAN_THREADS = 256;  // the finalising CTA's size, which the rounds assume
static_assert(RESCAN_ROUNDS * RESCAN_THREADS >= RESCAN_RANGE_VEC, "the rounds cover the range");

struct RescanSmem {
    float wsum[RESCAN_ROUNDS * 8];  // per (round, warp) totals
    int kmin;                       // first vector whose running mass crosses t
    int klast;                      // last vector with positive mass
    int found;
};

// The vectors covering columns [c0, c1) of a row, vector i starting at column a0 + i * VEC, a0
// being c0 rounded down to a 16-byte boundary (row points at column 0; rowflat is the row's first
// element in the flat logits array of `total` elements, whose base is mis elements past a 16-byte
// boundary): thread t loads vectors t + i * RESCAN_THREADS.  Whole aligned vectors are read even
// where they stick out of [c0, c1) (the weights mask those elements); only a vector that would
// reach outside the logits array is read element by element.
template <typename T>
__device__ __forceinline__ void load_range(const T *row, int64_t rowflat, int64_t total, int mis, int c0, int c1,
                                           uint4 (&w)[RESCAN_ROUNDS])
{
    constexpr int VEC = Elt<T>::VEC;
    const int a0 = c0 - (int)((rowflat + c0 + mis) % VEC);
    const int nvv = (c1 - a0 + VEC - 1) / VEC;
#pragma unroll
    for (int i = 0; i < RESCAN_ROUNDS; ++i) {
        const int k = threadIdx.x + i * RESCAN_THREADS;
        w[i] = make_uint4(0u, 0u, 0u, 0u);
        if (k < nvv) {
            const int col = a0 + k * VEC;
            const int64_t f = rowflat + col;
            w[i] = (f >= 0 && f + VEC <= total && SV_INB(f + VEC - 1, total, 401)) ? ldg_stream(row + col)
                                                                               : load_partial<T>(row, col, c0, c1);
        }
    }
}

// First column y of [c0, c1) at which cum0 + (running weight up to and including y) exceeds t;
// when none does (t = +inf asks for that), the last column with positive weight; -1 if no weight
// is positive.  Child tokens ex[0..ex_n) weigh 0.  w holds the range as load_range loads it; all
// RESCAN_THREADS threads of the CTA call it and get the result.  Per-round warp scans and one
// table of (round, warp) totals give every vector its running mass; the first crossing vector
// (or the last positive one) comes from shared-memory atomics, and its owner walks its VEC
// elements.  Three barriers, and one shared-memory atomic per warp.
template <typename T, bool FILT>
__device__ int rescan_range(int64_t rowflat, int mis, int c0, int c1, float cs, float mc, float thr, float t,
                            float cum0, const int *ex, int ex_n, const uint4 (&w)[RESCAN_ROUNDS], RescanSmem &S)
{
    constexpr int VEC = Elt<T>::VEC;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int nt = RESCAN_THREADS, nw = RESCAN_THREADS / 32;
    const int a0 = c0 - (int)((rowflat + c0 + mis) % VEC);
    const int nvv = (c1 - a0 + VEC - 1) / VEC;
    if (tid == 0) {
        S.kmin = INT_MAX;
        S.klast = -1;
    }
    float vs[RESCAN_ROUNDS], inc[RESCAN_ROUNDS];
#pragma unroll
    for (int i = 0; i < RESCAN_ROUNDS; ++i) {
        const int k = tid + i * nt;
        vs[i] = 0.f;
        if (k < nvv) {
            const int col = a0 + k * VEC;
            float e[VEC];
            vec_weights_plain<T, FILT>(w[i], col, c0, c1, cs, mc, thr, e);
            for (int x = 0; x < ex_n; ++x) {
                const int d = ex[x] - col;
#pragma unroll
                for (int j = 0; j < VEC; ++j)
                    if (j == d) e[j] = 0.f;
            }
            float p0 = (e[0] + e[1]) + (e[2] + e[3]);
            if (VEC == 8) p0 += (e[VEC - 4] + e[VEC - 3]) + (e[VEC - 2] + e[VEC - 1]);
            vs[i] = p0;
        }
        inc[i] = warp_incl_scan(vs[i], lane);
        if (lane == 31) S.wsum[i * 8 + warp] = inc[i];
    }
    __syncthreads();
    // Running mass before each (round, warp) block, in vector order.
    float pre[RESCAN_ROUNDS];
    float base = cum0;
#pragma unroll
    for (int i = 0; i < RESCAN_ROUNDS; ++i) {
        pre[i] = 0.f;
        for (int q = 0; q < nw; ++q) {
            if (q == warp) pre[i] = base;
            base += S.wsum[i * 8 + q];
        }
    }
    int kmin = INT_MAX, klast = -1;
#pragma unroll
    for (int i = 0; i < RESCAN_ROUNDS; ++i) {
        const int k = tid + i * nt;
        if (k < nvv && vs[i] > 0.f) {
            const float before = pre[i] + inc[i] - vs[i];
            if (kmin == INT_MAX && before + vs[i] > t) kmin = k;
            klast = k;
        }
    }
    // Reduce within the warp first: one shared-memory atomic per warp, not one per thread (every
    // thread past the crossing holds a candidate, and the same-address atomics serialise).
    kmin = __reduce_min_sync(0xffffffffu, kmin);
    klast = __reduce_max_sync(0xffffffffu, klast);
    if (lane == 0 && kmin != INT_MAX) atomicMin(&S.kmin, kmin);
    if (lane == 0 && klast >= 0) atomicMax(&S.klast, klast);
    __syncthreads();
    const bool last_mode = S.kmin == INT_MAX;
    const int kv = last_mode ? S.klast : S.kmin;
    if (kv < 0) {
        if (tid == 0) S.found = -1;
    } else if (kv % nt == tid) {
        const int i = kv / nt;
        float before = 0.f;
#pragma unroll
        for (int r = 0; r < RESCAN_ROUNDS; ++r)
            if (r == i) before = pre[r] + inc[r] - vs[r];
        const int col = a0 + kv * VEC;
        uint4 wv = w[0];
#pragma unroll
        for (int r = 1; r < RESCAN_ROUNDS; ++r)
            if (r == i) wv = w[r];
        float e[VEC];
        vec_weights_plain<T, FILT>(wv, col, c0, c1, cs, mc, thr, e);
        for (int x = 0; x < ex_n; ++x) {
            const int d = ex[x] - col;
#pragma unroll
            for (int j = 0; j < VEC; ++j)
                if (j == d) e[j] = 0.f;
        }
        float c = before;
        int found = -1, lp = -1;
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
            if (found < 0 && e[j] > 0.f) {
                lp = col + j;
                c += e[j];
                if (!last_mode && c > t) found = lp;
            }
        }
        // No element crossed (t = +inf, or rounding): the vector's last positive element.
        S.found = found >= 0 ? found : lp;
    }
    __syncthreads();
    return S.found;
}

// Locate step over one chunk of 32 records with masses m (in the row's reference): finds the
// first record where the running mass exceeds t, and tracks the last record with positive mass.
struct Locate {
    float cum = 0.f, before = 0.f, lp_before = 0.f;
    int found = -1, lastpos = -1;
};

__device__ __forceinline__ bool locate_chunk(Locate &Lc, float m, int c0, float t, int lane)
{
    const float incl = warp_incl_scan(m, lane);
    float excl = __shfl_up_sync(0xffffffffu, incl, 1);
    if (lane == 0) excl = 0.f;
    const unsigned hit = __ballot_sync(0xffffffffu, Lc.cum + incl > t);
    const unsigned pos = __ballot_sync(0xffffffffu, m > 0.f);
    if (pos) {
        const int lp = 31 - __clz(pos);
        Lc.lastpos = c0 + lp;
        Lc.lp_before = Lc.cum + __shfl_sync(0xffffffffu, excl, lp);
    }
    if (hit) {
        const int fl = __ffs(hit) - 1;
        Lc.found = c0 + fl;
        Lc.before = Lc.cum + __shfl_sync(0xffffffffu, excl, fl);
        return true;
    }
    Lc.cum += __shfl_sync(0xffffffffu, incl, 31);
    return false;
}

__device__ __forceinline__ float rec_mass(const float4 &r, float mc)
{
    return (r.y == 0.f) ? 0.f : r.y * ex2(r.x - mc);
}

}  // namespace sv
