// sv_draw.cuh -- block-wide inverse-CDF search over one segment of a row.
//
// The finalising CTA has already located the record (warp segment) in which the running sum
// of the draw's weights crosses the threshold t.  This file rescans only that segment, in
// ascending column order, and finds the first column whose running sum exceeds t.
//
// The segment is viewed as "groups" of GS consecutive columns; in round k thread tid owns
// group k * NT + tid, so the groups of one round are contiguous and in thread order.  KB
// rounds are loaded at once (one memory round trip), their totals reduced together to find the
// round that holds the crossing, and only that round is scanned thread by thread.
#pragma once

#include "sv_device.cuh"

namespace sv {

struct DrawSmem {
    float cum;          // weight before the part being scanned
    int found;          // column found (-1 while searching)
    int lastpos;        // last column with positive weight seen so far
    int first_thread;   // lowest thread whose inclusive sum crosses t
    float red[NW][16];  // per-warp partial totals of up to 16 rounds
    float tot[16];      // round totals
    float wpre[NW];     // exclusive warp prefixes of the scanned round
};

__device__ __forceinline__ float warp_incl_scan(float x, int lane)
{
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
    }
    return x;
}

__device__ __forceinline__ float warp_sum(float x)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

__device__ __forceinline__ int warp_max_int(int x)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x = max(x, __shfl_xor_sync(0xffffffffu, x, off));
    return x;
}

// Src provides:  using Raw = ...;  static constexpr int GS;
//   Raw prefetch(int64_t gi) const;                      // issue the loads of group gi
//   int weights(const Raw&, int64_t gi, float (&w)[GS]) const;  // weights; returns first column
// KB rounds per batch (<= 16).  All threads of the CTA must call.
template <int KB, typename Src>
__device__ void draw_span(const Src &src, int64_t ngroups, float t, DrawSmem &D)
{
    constexpr int GS = Src::GS;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int64_t gbase = 0; gbase < ngroups; gbase += (int64_t)KB * NT) {
        if (D.found >= 0) break;  // uniform: read after the barrier that ended the last batch
        typename Src::Raw raw[KB];
#pragma unroll
        for (int k = 0; k < KB; ++k) {
            const int64_t gi = gbase + (int64_t)k * NT + tid;
            if (gi < ngroups) raw[k] = src.prefetch(gi);
        }
        float own[KB];
        int lastpos = -1;
#pragma unroll
        for (int k = 0; k < KB; ++k) {
            own[k] = 0.f;
            const int64_t gi = gbase + (int64_t)k * NT + tid;
            if (gi < ngroups) {
                float w[GS];
                const int col0 = src.weights(raw[k], gi, w);
#pragma unroll
                for (int j = 0; j < GS; ++j) {
                    own[k] += w[j];
                    if (w[j] > 0.f) lastpos = col0 + j;
                }
            }
        }
        // Round totals and the last positive column.
#pragma unroll
        for (int k = 0; k < KB; ++k) {
            const float s = warp_sum(own[k]);
            if (lane == 0) D.red[warp][k] = s;
        }
        lastpos = warp_max_int(lastpos);
        if (lane == 0 && lastpos >= 0) atomicMax(&D.lastpos, lastpos);
        __syncthreads();
        if (tid < KB) {
            float s = 0.f;
            for (int w = 0; w < NW; ++w) s += D.red[w][tid];
            D.tot[tid] = s;
        }
        __syncthreads();
        float cum = D.cum;
        int kstar = -1;
#pragma unroll
        for (int k = 0; k < KB; ++k) {
            if (kstar < 0) {
                if (cum + D.tot[k] > t) kstar = k;
                else cum += D.tot[k];
            }
        }
        if (kstar < 0) {
            __syncthreads();  // everyone has read D.cum / D.tot
            if (tid == 0) D.cum = cum;
            __syncthreads();
            continue;
        }
        // Scan round kstar thread by thread.
        float mine = 0.f;
        typename Src::Raw rk = raw[0];
#pragma unroll
        for (int k = 0; k < KB; ++k) {
            if (k == kstar) {
                mine = own[k];
                rk = raw[k];
            }
        }
        const float incl_w = warp_incl_scan(mine, lane);
        float excl_w = __shfl_up_sync(0xffffffffu, incl_w, 1);
        if (lane == 0) excl_w = 0.f;
        if (lane == 31) D.wpre[warp] = incl_w;
        if (tid == 0) D.first_thread = NT;
        __syncthreads();
        if (warp == 0) {
            const float x = lane < NW ? D.wpre[lane] : 0.f;
            const float xi = warp_incl_scan(x, lane);
            float xe = __shfl_up_sync(0xffffffffu, xi, 1);
            if (lane == 0) xe = 0.f;
            __syncwarp();
            if (lane < NW) D.wpre[lane] = xe;
        }
        __syncthreads();
        const float incl = cum + (D.wpre[warp] + incl_w);
        const float excl = cum + (D.wpre[warp] + excl_w);
        // The warp's first crossing lane, then one shared-memory atomic per warp.
        const unsigned cross = __ballot_sync(0xffffffffu, incl > t);
        if (lane == 0 && cross) atomicMin(&D.first_thread, warp * 32 + __ffs(cross) - 1);
        __syncthreads();
        if (tid == D.first_thread) {
            const int64_t gi = gbase + (int64_t)kstar * NT + tid;
            float w[GS];
            const int col0 = src.weights(rk, gi, w);
            float c = excl;
            int found = -1, lastp = -1;
#pragma unroll
            for (int j = 0; j < GS; ++j) {
                if (found < 0 && w[j] > 0.f) {
                    lastp = col0 + j;
                    c += w[j];
                    if (c > t) found = col0 + j;
                }
            }
            D.found = found >= 0 ? found : lastp;
        }
        if (D.first_thread == NT && tid == 0) {
            // Rounding put the crossing past the round: keep searching after it.
            D.cum = cum + D.tot[kstar];
        }
        __syncthreads();
        if (D.first_thread == NT) {
            // Continue with the rounds after kstar in this batch, which were not accumulated.
            float c2 = D.cum;
            for (int k = kstar + 1; k < KB; ++k) c2 += D.tot[k];
            __syncthreads();
            if (tid == 0) D.cum = c2;
            __syncthreads();
        }
    }
}

}  // namespace sv
