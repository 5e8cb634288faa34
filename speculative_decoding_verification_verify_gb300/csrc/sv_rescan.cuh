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

__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gsrc)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                     (uint32_t)__cvta_generic_to_shared(smem_dst)),
                 "l"(gsrc)
                 : "memory");
}

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
    int first;       // lowest thread whose running weight crosses t
    int last;        // highest thread with positive weight
    int found;
};

// First column y of [c0, c1) at which cum0 + (running weight up to and including y) exceeds t;
// when none does (t = +inf asks for that), the last column with positive weight; -1 if no weight
// is positive.  Child tokens ex[0..ex_n) (sorted) weigh 0.  row points at column 0 of the row;
// rowflat is the row's first element in the flat logits array of `total` elements, whose base is
// mis elements past a 16-byte boundary.  stage holds RESCAN_STAGE_VEC shared vectors.  Every
// thread of the CTA calls it and gets the result.
template <typename T>
__device__ int block_rescan(const T *row, int64_t rowflat, int64_t total, int mis, int c0, int c1,
                            float cs, float mc, float t, float cum0, const int *ex, int ex_n,
                            uint4 *stage, RescanSmem &S)
{
    constexpr int VEC = Elt<T>::VEC;
    const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5, nw = nt >> 5;
    const int a0 = c0 - (int)((rowflat + c0 + mis) % VEC);  // aligned-down start column
    const int nvv = (c1 - a0 + VEC - 1) / VEC;
    // Whole aligned vectors are copied even where they stick out of [c0, c1) (the weights mask
    // those elements); only a vector that would reach outside the logits array is read element
    // by element.
    for (int i = tid; i < nvv; i += nt) {
        const int col = a0 + i * VEC;
        const int64_t f = rowflat + col;
        if (f >= 0 && f + VEC <= total) cp_async16(stage + i, row + col);
        else stage[i] = load_partial<T>(row, col, c0, c1);
    }
    if (tid == 0) {
        S.first = INT_MAX;
        S.last = -1;
        S.found = -1;
    }
    asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
    __syncthreads();
    // Each thread weighs a contiguous run of odd length (conflict-free 16-byte shared reads).
    const int per = ((nvv + nt - 1) / nt) | 1;
    const int k0 = min(tid * per, nvv), k1 = min(k0 + per, nvv);
    const int lc0 = a0 + k0 * VEC, lc1 = a0 + k1 * VEC;
    int e0 = 0;
    while (e0 < ex_n && ex[e0] < lc0) ++e0;
    int e1 = e0;
    while (e1 < ex_n && ex[e1] < lc1) ++e1;
    float own = 0.f;
    for (int k = k0; k < k1; ++k) {
        float e[VEC];
        vec_weights_ex<T>(stage[k], a0 + k * VEC, c0, c1, cs, mc, ex, e0, e1, e);
#pragma unroll
        for (int j = 0; j < VEC; ++j) own += e[j];
    }
    // Block scan of the thread totals.
    const float incl = warp_incl_scan(own, lane);
    if (lane == 31) S.wsum[warp] = incl;
    __syncthreads();
    const float ws = lane < nw ? S.wsum[lane] : 0.f;
    const float wi = warp_incl_scan(ws, lane);
    const float cum = cum0 + __shfl_sync(0xffffffffu, wi - ws, warp);
    if (cum + incl > t) atomicMin(&S.first, tid);
    if (own > 0.f) atomicMax(&S.last, tid);
    __syncthreads();
    const bool take_last = S.first == INT_MAX;
    const int who = take_last ? S.last : S.first;
    if (tid == who) {
        // Walk the run: the first crossing, or (take_last, or rounding) the last positive column.
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
                    if (!take_last && c > t) found = lp;
                }
            }
        }
        S.found = found >= 0 ? found : lp;
    }
    __syncthreads();
    return S.found;
}

}  // namespace sv
