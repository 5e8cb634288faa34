// sv_rescan.cuh -- the draw's block-wide rescan of one record segment, kept compact.
//
// The finalising CTA knows which warp segment of the stop row holds the crossing of v * Z.  It
// copies that segment into shared memory with cp.async (hardware-tracked, nothing spins), then
// one rolled pass gives each thread the weight of its contiguous share, one block scan orders
// the shares, and the thread whose share crosses the threshold walks it.  The code is small on
// purpose: it runs once per request on an SM whose instruction cache has never seen it.
#pragma once

#include "sv_device.cuh"

namespace sv {

constexpr int RESCAN_VEC = 4096;  // 16-byte vectors staged per pass (64 KB)
constexpr size_t RESCAN_SMEM_BYTES = (size_t)(RESCAN_VEC + 2) * 16;

struct RescanSmem {
    float wsum[NW];
    float cum;
    float total;
    int found;
    int lastpos;
    int first;
};

__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gsrc)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                     (uint32_t)__cvta_generic_to_shared(smem_dst)),
                 "l"(gsrc)
                 : "memory");
}

// Weights of one staged 16-byte vector whose first element has stage index i0 and column col0:
// 2^(x*cs - mc) for stage indices in [lo, hi) that are not excluded columns, else 0.  The
// cursor ep walks the sorted excluded columns (a thread's vectors come in ascending order).
template <typename T>
__device__ __forceinline__ void staged_weights(const uint4 &w, int i0, int lo, int hi, int col0,
                                               float cs, float mc, const int *ex, int ex_cnt,
                                               int &ep, float (&out)[Elt<T>::VEC])
{
    constexpr int VEC = Elt<T>::VEC;
    float x[VEC];
    Elt<T>::unpack(w, x);
#pragma unroll
    for (int j = 0; j < VEC; ++j) {
        const float e = ex2(fmaf(x[j], cs, -mc));
        out[j] = (i0 + j >= lo && i0 + j < hi) ? e : 0.f;
    }
    while (ep < ex_cnt && ex[ep] < col0) ++ep;
    for (int e = ep; e < ex_cnt && ex[e] < col0 + VEC; ++e) {
#pragma unroll
        for (int j = 0; j < VEC; ++j)
            if (col0 + j == ex[e]) out[j] = 0.f;
    }
}

// First column of [sg.c0, sg.c1) where cum0 + running weight exceeds t; the last column with
// positive weight if none does (t = +inf asks for that).  All threads of the CTA call it.
template <typename T, int NTR>
__device__ int rescan_segment(const T *row, const Seg &sg, float cs, float mc, float t, float cum0,
                              const int *ex, int ex_cnt, unsigned char *stage_bytes,
                              RescanSmem &R)
{
    constexpr int VEC = Elt<T>::VEC;
    constexpr int NWR = NTR / 32;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    T *stage = reinterpret_cast<T *>(stage_bytes);
    const int c0 = (int)sg.c0, c1 = (int)sg.c1, b0 = (int)sg.b0, b1 = (int)sg.b1;
    const int nbody = (b1 - b0) / VEC;
    const int npass = nbody > 0 ? (nbody + RESCAN_VEC - 1) / RESCAN_VEC : 1;
    if (tid == 0) {
        R.cum = cum0;
        R.found = -1;
        R.lastpos = -1;
    }
    __syncthreads();
#pragma unroll 1
    for (int pass = 0; pass < npass; ++pass) {
        const int v0 = pass * RESCAN_VEC;
        const int nv = min(RESCAN_VEC, nbody - v0 > 0 ? nbody - v0 : 0);
        const bool first = pass == 0, last = pass == npass - 1;
        const int cb0 = b0 + v0 * VEC;          // column at stage index VEC
        const int nhead = first ? b0 - c0 : 0;  // < VEC
        const int ntail = last ? c1 - b1 : 0;   // < VEC
        for (int v = tid; v < nv; v += NTR) cp_async16(stage + VEC + v * VEC, row + cb0 + v * VEC);
        if (tid < nhead) stage[VEC - nhead + tid] = row[c0 + tid];
        if (tid < ntail) stage[VEC + nv * VEC + tid] = row[b1 + tid];
        asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
        __syncthreads();
        const int lo = VEC - nhead, hi = VEC + nv * VEC + ntail;
        const int colbase = cb0 - VEC;          // column of stage index 0
        const uint4 *sv = reinterpret_cast<const uint4 *>(stage_bytes);
        const int nsv = (hi + VEC - 1) / VEC;   // stage vectors holding [lo, hi)
        const int per = (nsv + NTR - 1) / NTR;
        const int v0s = min(tid * per, nsv), v1s = min(v0s + per, nsv);
        int ep = 0, lastpos = -1;
        float own = 0.f;
#pragma unroll 1
        for (int v = v0s; v < v1s; ++v) {
            float w[VEC];
            staged_weights<T>(sv[v], v * VEC, lo, hi, colbase + v * VEC, cs, mc, ex, ex_cnt, ep, w);
#pragma unroll
            for (int j = 0; j < VEC; ++j) {
                if (w[j] > 0.f) lastpos = colbase + v * VEC + j;
                own += w[j];
            }
        }
        // Block scan of the shares.
        float incl = own;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += y;
        }
        if (lane == 31) R.wsum[warp] = incl;
        for (int off = 16; off > 0; off >>= 1) lastpos = max(lastpos, __shfl_xor_sync(0xffffffffu, lastpos, off));
        if (lane == 0 && lastpos >= 0) atomicMax(&R.lastpos, lastpos);
        if (tid == 0) R.first = NTR;
        __syncthreads();
        float wpre = 0.f, tot = 0.f;
        for (int w = 0; w < NWR; ++w) {
            if (w < warp) wpre += R.wsum[w];
            tot += R.wsum[w];
        }
        float exw = __shfl_up_sync(0xffffffffu, incl, 1);
        if (lane == 0) exw = 0.f;
        const float cum = R.cum;
        const float excl = cum + wpre + exw;
        if (cum + wpre + incl > t) atomicMin(&R.first, tid);
        __syncthreads();
        if (tid == R.first) {
            float c = excl;
            int found = -1, lp = -1, e2 = 0;
#pragma unroll 1
            for (int v = v0s; v < v1s && found < 0; ++v) {
                float w[VEC];
                staged_weights<T>(sv[v], v * VEC, lo, hi, colbase + v * VEC, cs, mc, ex, ex_cnt, e2, w);
#pragma unroll
                for (int j = 0; j < VEC; ++j) {
                    if (found < 0 && w[j] > 0.f) {
                        lp = colbase + v * VEC + j;
                        c += w[j];
                        if (c > t) found = lp;
                    }
                }
            }
            R.found = found >= 0 ? found : lp;
        }
        if (tid == 0) R.total = cum + tot;
        __syncthreads();
        if (R.found >= 0) break;
        if (tid == 0) R.cum = R.total;
        __syncthreads();
    }
    return R.found >= 0 ? R.found : R.lastpos;
}

}  // namespace sv
