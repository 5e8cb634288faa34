// sv_rescan.cuh -- the finalising CTA draws a token from a short column range of a logit row.
//
// The finalising kernel knows which record of the streaming pass holds the crossing of the draw
// threshold t, and the mass before that record.  The record covers a column range of at most
// SUB_VEC 16-byte vectors (plus an unaligned head and tail), so the CTA copies that range into
// shared memory with cp.async (every copy in flight at once, completion tracked by the
// hardware), each thread weighs a contiguous run of a few vectors as the streaming pass did, a
// block scan of the thread totals picks the thread that holds the crossing, and that thread walks
// its run.  Loops stay short: this code runs once per request on an SM whose instruction cache
// has not seen it.
#pragma once

#include <climits>

#include "sv_device.cuh"
#include "sv_draw.cuh"

namespace sv {

// Shared-memory vectors the CTA stages: the range holds at most SUB_VEC aligned vectors plus a
// partial one at each end.
constexpr int RESCAN_STAGE_VEC = SUB_VEC + 2;

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

// Weights of one vector at column col with no excluded column in it; elements outside [c0, c1)
// weigh 0 (only the range's first and last vectors have such elements).
template <typename T>
__device__ __forceinline__ void vec_weights_plain(const uint4 &w, int col, int c0, int c1, float cs,
                                                  float mc, float (&out)[Elt<T>::VEC])
{
    constexpr int VEC = Elt<T>::VEC;
    float x[VEC];
    Elt<T>::unpack(w, x);
#pragma unroll
    for (int j = 0; j < VEC; ++j) out[j] = ex2(fmaf(x[j], cs, -mc));
    if (col < c0 || col + VEC > c1) {
#pragma unroll
        for (int j = 0; j < VEC; ++j)
            if (col + j < c0 || col + j >= c1) out[j] = 0.f;
    }
}

// The same with the excluded columns ex[e0..e1) (sorted) of this lane's run zeroed as well.
template <typename T>
__device__ __forceinline__ void vec_weights_ex(const uint4 &w, int col, int c0, int c1, float cs,
                                               float mc, const int *ex, int e0, int e1,
                                               float (&out)[Elt<T>::VEC])
{
    constexpr int VEC = Elt<T>::VEC;
    vec_weights_plain<T>(w, col, c0, c1, cs, mc, out);
    for (int e = e0; e < e1; ++e) {
        const int d = ex[e] - col;
#pragma unroll
        for (int j = 0; j < VEC; ++j)
            if (j == d) out[j] = 0.f;
    }
}

struct RescanSmem {
    float wsum[32];  // per-warp totals
    int found;
};

// Copy the vectors covering columns [c0, c1) of a row into stage: vector i starts at column
// a0 + i*VEC, a0 being c0 rounded down to a 16-byte boundary (row points at column 0; rowflat is
// the row's first element in the flat logits array of `total` elements, whose base is mis
// elements past a 16-byte boundary).  Whole aligned vectors are copied even where they stick out
// of [c0, c1) (the weights mask those elements); only a vector that would reach outside the
// logits array is read element by element.  Threads t = 0..nt-1 share the copies; each thread
// commits its cp.async group and must wait for it before the stage is read.
template <typename T>
__device__ __forceinline__ void stage_range(const T *row, int64_t rowflat, int64_t total, int mis, int c0,
                                            int c1, uint4 *stage, int t, int nt)
{
    constexpr int VEC = Elt<T>::VEC;
    const int a0 = c0 - (int)((rowflat + c0 + mis) % VEC);
    const int nvv = (c1 - a0 + VEC - 1) / VEC;
    for (int i = t; i < nvv; i += nt) {
        const int col = a0 + i * VEC;
        const int64_t f = rowflat + col;
        if (f >= 0 && f + VEC <= total) cp_async16(stage + i, row + col);
        else stage[i] = load_partial<T>(row, col, c0, c1);
    }
    cp_async_commit();
}

// First column y of [c0, c1) at which cum0 + (running weight up to and including y) exceeds t;
// when none does (t = +inf asks for that), the last column with positive weight; -1 if no weight
// is positive.  Child tokens ex[0..ex_n) (sorted) weigh 0.  stage holds the range as stage_range
// laid it out, visible to every thread.  Every thread of the CTA calls it and gets the result.
// Threads take runs of at most RUN_MAX vectors; the warp whose prefix crosses t (or, with none,
// the last warp with positive weight) finds the thread and the column, so two barriers suffice.
constexpr int RUN_MAX = 3;  // vectors per thread: (SUB_VEC + 2) / NT_FIN rounded up to odd

template <typename T>
__device__ int rescan_staged(int64_t rowflat, int mis, int c0, int c1, float cs, float mc, float t,
                             float cum0, const int *ex, int ex_n, const uint4 *stage, RescanSmem &S)
{
    constexpr int VEC = Elt<T>::VEC;
    const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5, nw = nt >> 5;
    const int a0 = c0 - (int)((rowflat + c0 + mis) % VEC);
    const int nvv = (c1 - a0 + VEC - 1) / VEC;
    // Each thread weighs a contiguous run of odd length (conflict-free 16-byte shared reads).
    const int per = ((nvv + nt - 1) / nt) | 1;
    const int k0 = min(tid * per, nvv), k1 = min(k0 + per, nvv);
    const int lc0 = a0 + k0 * VEC, lc1 = a0 + k1 * VEC;
    int e0 = 0;
    while (e0 < ex_n && ex[e0] < lc0) ++e0;
    int e1 = e0;
    while (e1 < ex_n && ex[e1] < lc1) ++e1;
    float vs[RUN_MAX];
    float own = 0.f;
    if (per <= RUN_MAX) {
#pragma unroll
        for (int i = 0; i < RUN_MAX; ++i) {
            vs[i] = 0.f;
            if (k0 + i < k1) {
                float e[VEC];
                vec_weights_ex<T>(stage[k0 + i], a0 + (k0 + i) * VEC, c0, c1, cs, mc, ex, e0, e1, e);
                float p0 = (e[0] + e[1]) + (e[2] + e[3]);
                if (VEC == 8) p0 += (e[VEC - 4] + e[VEC - 3]) + (e[VEC - 2] + e[VEC - 1]);
                vs[i] = p0;
            }
            own += vs[i];
        }
    } else {
        for (int k = k0; k < k1; ++k) {
            float e[VEC];
            vec_weights_ex<T>(stage[k], a0 + k * VEC, c0, c1, cs, mc, ex, e0, e1, e);
#pragma unroll
            for (int j = 0; j < VEC; ++j) own += e[j];
        }
    }
    // Warp totals, then every warp knows its prefix.
    const float incl = warp_incl_scan(own, lane);
    if (lane == 31) S.wsum[warp] = incl;
    __syncthreads();
    const float ws = lane < nw ? S.wsum[lane] : 0.f;
    const float wi = warp_incl_scan(ws, lane);
    const unsigned wcross = __ballot_sync(0xffffffffu, lane < nw && cum0 + wi > t);
    const unsigned wpos = __ballot_sync(0xffffffffu, lane < nw && ws > 0.f);
    const bool take_last = wcross == 0;
    const int wsel = take_last ? (wpos ? 31 - __clz(wpos) : -1) : __ffs(wcross) - 1;
    if (warp == wsel) {
        const float cum = cum0 + __shfl_sync(0xffffffffu, wi - ws, warp);
        const unsigned hit = __ballot_sync(0xffffffffu, !take_last && cum + incl > t);
        const unsigned pos = __ballot_sync(0xffffffffu, own > 0.f);
        // The crossing thread, or (take_last, or rounding) the warp's last positive thread.
        const bool last_mode = hit == 0;
        const int who = last_mode ? 31 - __clz(pos) : __ffs(hit) - 1;
        if (lane == who) {
            float c = cum + incl - own;
            int found = -1, lp = -1;
            for (int k = k0; k < k1 && found < 0; ++k) {
                const int col = a0 + k * VEC;
                float e[VEC];
                vec_weights_ex<T>(stage[k], col, c0, c1, cs, mc, ex, e0, e1, e);
#pragma unroll
                for (int j = 0; j < VEC; ++j) {
                    if (found < 0 && e[j] > 0.f) {
                        lp = col + j;
                        c += e[j];
                        if (!last_mode && c > t) found = lp;
                    }
                }
            }
            S.found = found >= 0 ? found : lp;
        }
    } else if (wsel < 0 && tid == 0) {
        S.found = -1;
    }
    __syncthreads();
    return S.found;
}

}  // namespace sv
